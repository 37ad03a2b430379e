"""The C ABI's calls can be captured in a CUDA graph: the forward, the
backward (whose tensor-core grid is a programmatic dependent launch of its
D pass) and split-KV decoding (whose combine kernel is one of its partial
kernel), each replayed from a graph, give the bit-identical results of the
same calls made eagerly.  Each call is made once eagerly before capture
(per-device setup such as the shared-memory limits happens then)."""
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import seeded_inputs
from gpu_common import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream())
    return g


def test_forward_and_backward_in_a_graph():
    B, H, N, d = 1, 4, 700, 128
    q, k, v = (t.cuda() for t in seeded_inputs.make_qkv(B, H, N, d, "bf16", 1.0, seed=5))
    do = seeded_inputs.make_dout(B, H, N, d, "bf16", seed=5).cuda()
    o_ref, l_ref = fa.attention_forward(q, k, v, causal=True)
    g_ref = fa.attention_backward(q, k, v, o_ref, l_ref, do, causal=True)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    code = fa.dtype_code(q.dtype)
    scale = 1.0 / d ** 0.5

    def step(st):
        assert fa.fa_fwd(q, k, v, o, lse, B, H, N, d, 1, scale, code, st) == fa.FA_OK
        assert fa.fa_bwd(q, k, v, o, lse, do, gq, gk, gv, delta, B, H, N, d, 1, scale, code,
                         st) == fa.FA_OK

    g = capture(step)
    for t in (o, gq, gk, gv):
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    for a, b in zip((gq, gk, gv), g_ref):
        assert torch.equal(a, b)


def test_decode_in_a_graph():
    B, H, Nq, Nk, d = 2, 4, 1, 20000, 64
    q, k, v = (t.cuda() for t in seeded_inputs.make_decode(B, H, Nq, Nk, d, "fp16", seed=6))
    o_ref, l_ref = fa.attention_decode(q, k, v, causal=True)
    nbytes = fa.fa_decode_workspace_size(B, H, Nq, Nk, d)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    o, lse = torch.empty_like(q), torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    code = fa.dtype_code(q.dtype)

    def step(st):
        assert fa.fa_decode(q, k, v, o, lse, B, H, Nq, Nk, d, 1, 1.0 / d ** 0.5, code, ws, nbytes,
                            st) == fa.FA_OK

    g = capture(step)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
