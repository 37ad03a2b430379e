"""Failure detection without a GPU fault: a bounded wait that runs out.

fa_watchdog_selftest launches a one-thread kernel whose wait — the bounded
wait every kernel of the library uses — is on a barrier nothing completes.
After its budget the wait records a timeout and its site in the status word
and the kernel returns.  fa_status must report FA_ERR_TIMEOUT with that
site, clear the word, and the next real call must be correct (the context
stays usable).  No trap, assert, bad address or endless loop is involved.
"""
import time

import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
from gpu_common import compare, default_scale, make, oracle_full, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_wait_runs_out_is_reported_and_the_context_stays_usable():
    assert fa.fa_status()[0] == fa.FA_OK             # nothing pending from earlier tests
    t0 = time.perf_counter()
    assert fa.fa_watchdog_selftest(2_000_000) == fa.FA_OK   # 2 ms budget
    code, word = fa.fa_status()
    elapsed = time.perf_counter() - t0
    assert code == fa.FA_ERR_TIMEOUT, (code, hex(word))
    assert word & 1 and (word >> 8) & 0xff == 31, hex(word)
    assert elapsed < 5.0                              # the wait ended by itself
    assert fa.fa_status()[0] == fa.FA_OK             # fa_status cleared the word
    for d, causal in ((128, False), (64, True)):
        q, k, v = make(1, 2, 640, d, "bf16", seed=50 + d)
        o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal)
        torch.cuda.synchronize()
        assert fa.fa_status()[0] == fa.FA_OK
        o_ref, lse_ref = oracle_full(q, k, v, causal, default_scale(d))
        compare(o.cpu(), lse.cpu(), o_ref, lse_ref, "bf16", f"after the self-test d={d}")


def test_selftest_argument_errors():
    assert fa.fa_watchdog_selftest(0) == fa.FA_ERR_SHAPE
    assert fa.fa_watchdog_selftest(2_000_000_000) == fa.FA_ERR_SHAPE
