"""moe_permute_static -- the permutation for callers that cannot allocate
device memory (plug-in hosts with no allocator, processes whose device memory
is all held by a framework pool) -- must give exactly what moe_permute gives
with a caller workspace.  Two calls in a row with different shapes check that
the fixed scratch it shares across calls does not carry anything over.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import gen

pytestmark = pytest.mark.gpu

OUT = ("counts_raw", "counts", "offsets", "row_of_slot", "slot_of_row", "x_perm")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def _buffers(T, d, E, k):
    z = lambda n: torch.full((n,), -3, dtype=torch.int32, device="cuda")  # noqa: E731
    return {"counts_raw": z(E), "counts": z(E), "offsets": z(E + 1), "row_of_slot": z(T * k),
            "slot_of_row": z(T * k), "x_perm": torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")}


def _run(B, static, x, idx, T, d, E, k, cap):
    o = _buffers(T, d, E, k)
    if static:
        B.moe_permute_static(x, idx, T, d, E, k, cap, o["counts_raw"], o["counts"], o["offsets"], o["row_of_slot"],
                             o["slot_of_row"], o["x_perm"])
    else:
        ws_bytes = B.moe_workspace_size(T, d, E, k, 128, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        B.moe_permute(x, idx, T, d, E, k, cap, o["counts_raw"], o["counts"], o["offsets"], o["row_of_slot"],
                      o["slot_of_row"], o["x_perm"], ws, ws_bytes)
    torch.cuda.synchronize()
    return o


def _case(T, E, k, d, tensor):
    l = gen.random_logits(T, E, tensor=tensor)
    l[:, :2] += 1.5  # two hot experts
    idx, _ = orc.route_topk(l, k)
    x = torch.from_numpy(gen.normal_bf16(tensor + 1, (T, d)).view(np.int16)).cuda().view(torch.bfloat16)
    return x, torch.from_numpy(idx).cuda()


def test_static_scratch_matches_workspace_version_on_two_calls_in_a_row(B):
    cases = [(3000, 64, 4, 256, 40), (1500, 128, 8, 128, 0)]   # (T, E, k, d, capacity)
    for n, (T, E, k, d, cap) in enumerate(cases):
        x, idx = _case(T, E, k, d, tensor=500 + 10 * n)
        ref = _run(B, False, x, idx, T, d, E, k, cap)
        got = _run(B, True, x, idx, T, d, E, k, cap)
        R = int(ref["offsets"][-1].item())
        for key in OUT:
            a, b = ref[key], got[key]
            if key in ("slot_of_row", "x_perm"):
                a, b = a[:R], b[:R]
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b), (n, key)
    assert B.moe_device_status() == 0


def test_static_scratch_rejects_shapes_beyond_its_size(B):
    """The size check comes before any device access: the pointers are never
    dereferenced."""
    T, E, k, d = 1 << 20, 256, 8, 64    # needs ~48 MiB of scratch, more than the fixed 4 MiB
    p = 1 << 12                         # stand-in addresses, 16-byte aligned
    with pytest.raises(B.MoEError) as ei:
        B.moe_permute_static(p, p, T, d, E, k, 0, p, p, p, p, p, p)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
