"""The unit order of the persistent forward kernels changes which CTA
computes which query block, never a result: outputs are bit-identical for
every group size fa_set_unit_group forces (including one above B*H, which
is clamped) and the automatic choice, for square, kv and packed calls."""
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import seeded_inputs
from gpu_common import require_gpu

pytestmark = pytest.mark.gpu

GROUPS = [1, 3, 7, 1000, 0]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    fa.fa_set_unit_group(0)


def run_each_group(fn):
    outs = []
    for g in GROUPS:
        assert fa.fa_set_unit_group(g) == fa.FA_OK
        outs.append([t.clone() for t in fn()])
        torch.cuda.synchronize()
    fa.fa_set_unit_group(0)
    assert fa.fa_status()[0] == fa.FA_OK
    for g, o in zip(GROUPS[1:], outs[1:]):
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b), f"group {g} differs from group {GROUPS[0]}"


@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False)])
def test_square_invariant(d, causal):
    q, k, v = (t.cuda() for t in seeded_inputs.make_qkv(2, 5, 1500, d, "bf16", 1.0, seed=d + causal))
    run_each_group(lambda: fa.attention_forward(q, k, v, causal=causal))


def test_kv_invariant():
    q, k, v = (t.cuda() for t in seeded_inputs.make_decode(3, 4, 700, 2100, 128, "fp16", seed=3))
    sl = torch.tensor([2100, 999, 5], dtype=torch.int32, device="cuda")
    run_each_group(lambda: fa.attention_forward_kv(q, k, v, causal="bottom_right"))
    run_each_group(lambda: fa.attention_forward_kv(q, k, v, causal="upper_left", seqlens_k=sl))


def test_varlen_invariant():
    lens = [900, 17, 1300, 256]
    q, k, v, cq, ck = seeded_inputs.make_varlen(lens, lens, 3, 64, "bf16", seed=4)
    q, k, v, cq, ck = (t.cuda() for t in (q, k, v, cq, ck))
    run_each_group(lambda: fa.attention_forward_varlen(q, k, v, cq, ck, max(lens),
                                                       causal="upper_left"))
