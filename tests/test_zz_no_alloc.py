"""fa_fwd_static, the forward entry point that allocates nothing.

Callers that only hold raw device pointers (no allocator of their own), or
that must not call cudaMalloc on their path, use fa_fwd_static: its scratch
is a fixed device array inside the library.  This test calls it through the
C ABI twice in a row and checks both outputs against fa_fwd_ws run with a
workspace the test allocates, within the tolerances of the other GPU tests.
The first two shapes leave a partial last round on a 152-SM GPU, so they
run the split tail through the library's array; the third fills whole
rounds and needs no scratch.  Free device memory must not move across the
second call.  It sits in a file of its own that pytest collects last, and
passes both on its own in a fresh process and after the other tests.
"""
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
from gpu_common import LSE_TOL, TOL, default_scale, make, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,dtype,splits", [
    (1, 16, 4096, 128, "bf16", True),   # 256 units on 152 SMs: the last round is split
    (1, 40, 1024, 64, "fp16", True),    # tail pieces of a single key tile
    (1, 3, 500, 64, "bf16", False),     # no partial round: no scratch needed
])
def test_static_scratch_matches_workspace_entry_point(B, H, N, d, dtype, splits):
    require_gpu()
    if splits and torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the split cases are sized for a 152-SM GPU")
    q, k, v = (t.cuda() for t in make(B, H, N, d, dtype, q_std=2.0, seed=77 + N))
    scale = default_scale(d)
    code = fa.dtype_code(q.dtype)
    stream = torch.cuda.current_stream()
    need = fa.fa_fwd_workspace_size(B, H, N, d, False)
    assert (need > 0) == splits, f"workspace {need} bytes"

    # reference: the existing entry point with a workspace allocated here
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    ws = fa.make_workspace(B, H, N, d, False)
    ws_bytes = 0 if ws is None else ws.numel()
    assert fa.fa_fwd_ws(q, k, v, o_ref, lse_ref, B, H, N, d, False, scale, code, ws, ws_bytes,
                        stream) == fa.FA_OK

    outs = [(torch.full_like(q, float("nan")),
             torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda"))
            for _ in range(2)]
    torch.cuda.synchronize()
    free_before = None
    for call, (o, lse) in enumerate(outs):   # two calls in a row share the library's scratch
        if call == 1:
            free_before = torch.cuda.mem_get_info()[0]
        assert fa.fa_fwd_static(q, k, v, o, lse, B, H, N, d, False, scale, code,
                                stream) == fa.FA_OK
        torch.cuda.synchronize()
        if call == 1:
            moved = abs(torch.cuda.mem_get_info()[0] - free_before)
            assert moved <= 2 << 20, f"free device memory moved by {moved} bytes"
        assert fa.fa_status()[0] == fa.FA_OK
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        err = (o.double() - o_ref.double()).abs()
        assert err.max().item() <= TOL[dtype][0], f"call {call}: max|dO| {err.max().item():.3e}"
        assert err.mean().item() <= TOL[dtype][1]
        assert (lse - lse_ref).abs().max().item() <= LSE_TOL
