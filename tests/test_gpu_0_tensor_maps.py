"""The weight-gradient GEMMs read each expert's rows through tensor maps
patched on the device (base address and row extent re-set per group).  This
file sorts before every test that runs those GEMMs: the patched maps must be
byte-identical to the maps the CUDA driver's encoder gives for the same
sub-matrices (empty, one-row and ragged groups)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_device_patched_group_maps_match_the_driver_encoding():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding as B
    assert B.moe_selftest_group_maps() == B.MOE_OK
