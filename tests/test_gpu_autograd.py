"""The torch.autograd wrappers route to the C ABI: gradients taken through
autograd are bit-identical to calling the backward entry points directly
with the same upstream gradient (square, with dropout, kv, packed)."""
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import seeded_inputs
from gpu_common import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def leaves(*ts):
    return [t.cuda().requires_grad_(True) for t in ts]


@pytest.mark.parametrize("dropout_p", [0.0, 0.2])
def test_square(dropout_p):
    q, k, v = leaves(*seeded_inputs.make_qkv(1, 3, 500, 64, "bf16", 1.0, seed=21))
    w = seeded_inputs.make_dout(1, 3, 500, 64, "bf16", seed=21).cuda()
    o, lse = fa.flash_attention(q, k, v, causal=True, dropout_p=dropout_p, seed=9, offset=4)
    (o.float() * w.float()).sum().backward()
    qd, kd, vd = q.detach(), k.detach(), v.detach()
    if dropout_p:
        o2, l2 = fa.attention_forward_dropout(qd, kd, vd, dropout_p, 9, 4, causal=True)
        g = fa.attention_backward_dropout(qd, kd, vd, o2, l2, w, dropout_p, 9, 4, causal=True)
    else:
        o2, l2 = fa.attention_forward(qd, kd, vd, causal=True)
        g = fa.attention_backward(qd, kd, vd, o2, l2, w, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o2) and torch.equal(lse, l2)
    for a, b in zip((q.grad, k.grad, v.grad), g):
        assert torch.equal(a, b)


def test_kv():
    q, k, v = leaves(*seeded_inputs.make_decode(2, 2, 200, 700, 128, "fp16", seed=22))
    w = seeded_inputs.make_dout(2, 2, 200, 128, "fp16", seed=22).cuda()
    sl = torch.tensor([700, 333], dtype=torch.int32, device="cuda")
    o, lse = fa.flash_attention_kv(q, k, v, causal="bottom_right", seqlens_k=sl)
    (o.float() * w.float()).sum().backward()
    qd, kd, vd = q.detach(), k.detach(), v.detach()
    o2, l2 = fa.attention_forward_kv(qd, kd, vd, causal="bottom_right", seqlens_k=sl)
    g = fa.attention_backward_kv(qd, kd, vd, o2, l2, w, causal="bottom_right", seqlens_k=sl)
    torch.cuda.synchronize()
    for a, b in zip((q.grad, k.grad, v.grad), g):
        assert torch.equal(a, b)


def test_varlen():
    lens_q, lens_k = [100, 300, 7], [400, 300, 50]
    q, k, v, cq, ck = seeded_inputs.make_varlen(lens_q, lens_k, 2, 64, "bf16", seed=23)
    q, k, v = leaves(q, k, v)
    cq, ck = cq.cuda(), ck.cuda()
    w = torch.randn(q.shape, generator=torch.Generator("cpu").manual_seed(23)).to(q.dtype).cuda()
    o, lse = fa.flash_attention_varlen(q, k, v, cq, ck, 300, 400, causal="bottom_right")
    (o.float() * w.float()).sum().backward()
    qd, kd, vd = q.detach(), k.detach(), v.detach()
    o2, l2 = fa.attention_forward_varlen(qd, kd, vd, cq, ck, 300, causal="bottom_right")
    g = fa.attention_backward_varlen(qd, kd, vd, o2, l2, w, cq, ck, 300, 400, causal="bottom_right")
    torch.cuda.synchronize()
    for a, b in zip((q.grad, k.grad, v.grad), g):
        assert torch.equal(a, b)
