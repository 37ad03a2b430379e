"""The Python binding's argument checks (CPU only): each wrapper rejects a
dtype mix, a wrong rank or shape, host tensors, non-contiguous tensors and
unknown causal modes with TypeError or ValueError before anything reaches
the C ABI, so these run without a GPU."""
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa


def t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def test_forward_kv_checks():
    q, k = t(1, 2, 8, 64), t(1, 2, 16, 64)
    with pytest.raises(TypeError):
        fa.attention_forward_kv(q, k, t(1, 2, 16, 64, dtype=torch.float16))
    with pytest.raises(ValueError):
        fa.attention_forward_kv(q, k, t(1, 2, 15, 64))          # k, v lengths differ
    with pytest.raises(ValueError):
        fa.attention_forward_kv(q, t(1, 3, 16, 64), t(1, 3, 16, 64))   # heads differ
    with pytest.raises(ValueError):
        fa.attention_forward_kv(q, t(1, 2, 16, 128), t(1, 2, 16, 128))  # widths differ
    with pytest.raises(ValueError):
        fa.attention_forward_kv(q, k, k)                        # host tensors
    with pytest.raises(ValueError):
        fa.attention_forward_kv(q[0], k[0], k[0])               # rank


def test_forward_varlen_checks():
    q, k = t(10, 2, 64), t(20, 2, 64)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(TypeError):
        fa.attention_forward_varlen(q, k, t(20, 2, 64, dtype=torch.float16), cu, cu, 10)
    with pytest.raises(ValueError):
        fa.attention_forward_varlen(t(1, 10, 2, 64), k, k, cu, cu, 10)   # rank
    with pytest.raises(ValueError):
        fa.attention_forward_varlen(q, t(20, 3, 64), t(20, 3, 64), cu, cu, 10)
    with pytest.raises(ValueError):
        fa.attention_forward_varlen(q, k, k, cu, cu, 10)                 # host tensors


def test_backward_checks():
    q = t(1, 2, 8, 64)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(TypeError):
        fa.attention_backward(q, q, q, q, lse, t(1, 2, 8, 64, dtype=torch.float16))
    with pytest.raises(ValueError):
        fa.attention_backward(q, q, q, q, torch.zeros(1, 2, 7), q)         # lse shape
    with pytest.raises(ValueError):
        fa.attention_backward(q, q, q, q, lse.double(), q)                 # lse dtype
    with pytest.raises(ValueError):
        fa.attention_backward(q, q, q, q, lse, q)                          # host tensors
    with pytest.raises(ValueError):
        fa.attention_backward_kv(q, t(1, 2, 9, 64), t(1, 2, 9, 64), q, lse, q, causal="middle")
    with pytest.raises(ValueError):
        fa.attention_backward_kv(q, t(1, 2, 9, 64), t(1, 2, 9, 64), t(1, 2, 9, 64), lse, q)
    with pytest.raises(ValueError):
        fa.attention_backward_dropout(q, q, q, q, torch.zeros(2, 8), q, 0.1, 0, 0)


def test_backward_onepass_checks():
    q = t(1, 2, 8, 64)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(TypeError):
        fa.attention_backward_onepass(q, q, q, q, lse, t(1, 2, 8, 64, dtype=torch.float16))
    with pytest.raises(ValueError):
        fa.attention_backward_onepass(q, q, q, q, torch.zeros(1, 2, 7), q)   # lse shape
    with pytest.raises(ValueError):
        fa.attention_backward_onepass(q, q, q, q, lse.double(), q)           # lse dtype
    with pytest.raises(ValueError):
        fa.attention_backward_onepass(q, t(1, 2, 9, 64), q, q, lse, q)       # shapes differ
    with pytest.raises(ValueError):
        fa.attention_backward_onepass(q, q, q, q, lse, q, dropout_p=0.1)     # host tensors


def test_backward_varlen_checks():
    q, k = t(10, 2, 64), t(20, 2, 64)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    lse = torch.zeros(2, 10)
    with pytest.raises(ValueError):
        fa.attention_backward_varlen(q, k, k, q, torch.zeros(10, 2), q, cu, cu, 10, 20)  # lse
    with pytest.raises(ValueError):
        fa.attention_backward_varlen(q, k, k, q, lse, q, cu, cu, 10, 20, causal="x")
    with pytest.raises(ValueError):
        fa.attention_backward_varlen(q, k, k, q, lse, q, cu, cu, 10, 20)   # host tensors


def test_dropout_forward_checks():
    q = t(1, 2, 8, 64)
    with pytest.raises(TypeError):
        fa.attention_forward_dropout(q, q, t(1, 2, 8, 64, dtype=torch.float16), 0.1, 0, 0)
    with pytest.raises(ValueError):
        fa.attention_forward_dropout(q, t(1, 2, 9, 64), t(1, 2, 9, 64), 0.1, 0, 0)
    with pytest.raises(ValueError):
        fa.attention_forward_dropout(q, q, q, 0.1, 0, 0)                    # host tensors


def test_causal_modes_table():
    assert fa.CAUSAL_MODES == {None: 0, False: 0, "upper_left": 1, "bottom_right": 2}
