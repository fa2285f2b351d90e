"""Bounded waits: a pipeline wait made to expire on purpose (PAFP8_WAIT_CYCLES
set to one cycle, so the first wait for a page that has not landed gives up).
The kernels record PAFP8_ERR_TIMEOUT, wind down after their own copies and
MMAs in flight have finished, and return; the next run on the same workspace
with the default bound is clean and matches the oracle.  Nothing here faults
or hangs the GPU: every wait is bounded, and the final waits for in-flight
work keep the long bound."""
from __future__ import annotations

import pytest

import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import DeviceBatch, assert_close
from paged_attention_fp8_gb300.workloads import make_batch, workload

pytestmark = pytest.mark.gpu


def _batch(which):
    if which == "decode":
        return workload(1)
    if which == "decode_split":
        return make_batch([17, 900, 2500], num_qo_heads=32, num_kv_heads=8, seed=41)
    if which == "prefill_bf16":
        return make_batch([40, 300, 700], [40, 129, 256], num_qo_heads=32, num_kv_heads=8, seed=42)
    if which == "prefill_fp8":
        return make_batch([256, 300], [256, 129], num_qo_heads=32, num_kv_heads=8, q_dtype="e4m3fn",
                          kv_dtype="e4m3fn", o_dtype="bf16", seed=43)
    if which == "prefill_2byte_cache":
        return make_batch([40, 300], [40, 129], num_qo_heads=16, num_kv_heads=4, q_dtype="bf16",
                          kv_dtype="bf16", o_dtype="bf16", seed=44)
    raise ValueError(which)


@pytest.mark.parametrize("which", ["decode", "decode_split", "prefill_bf16", "prefill_fp8",
                                   "prefill_2byte_cache"])
def test_expired_wait_is_reported_and_the_next_run_is_clean(cuda_device, monkeypatch, which):
    b = _batch(which)
    db = DeviceBatch(b, cuda_device, num_ctas=8)
    monkeypatch.delenv("PAFP8_DEBUG", raising=False)
    monkeypatch.setenv("PAFP8_WAIT_CYCLES", "1")
    db.run()
    with pytest.raises(pa.Pafp8Error) as ei:
        db.plan.device_status(db.ws)
    assert ei.value.status == 6, str(ei.value)  # PAFP8_ERR_TIMEOUT
    monkeypatch.delenv("PAFP8_WAIT_CYCLES")
    db.o.fill_(float("nan"))
    db.lse.fill_(float("nan"))
    db.run()
    o, lse = db.result()  # raises unless the status word is clean
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, f"{which} after an expired wait")


def test_expired_wait_surfaces_at_the_call_in_debug_mode(cuda_device, monkeypatch):
    b = _batch("decode")
    db = DeviceBatch(b, cuda_device)
    monkeypatch.setenv("PAFP8_WAIT_CYCLES", "1")
    monkeypatch.setenv("PAFP8_DEBUG", "1")
    with pytest.raises(pa.Pafp8Error) as ei:
        db.run()
    assert ei.value.status == 6
    monkeypatch.delenv("PAFP8_WAIT_CYCLES")
    db.run()  # OK under PAFP8_DEBUG: the status word was read and cleared
    monkeypatch.setenv("PAFP8_DEBUG", "0")
    o, lse = db.result()
    ro, rl = oracle_on(b)
    assert_close(o, lse, ro, rl, "decode after an expired wait (debug mode)")


def test_wait_setting_is_ignored_unless_a_positive_integer(cuda_device, monkeypatch):
    b = _batch("decode")
    db = DeviceBatch(b, cuda_device)
    for bad in ("0", "-5", "abc", "12x", ""):
        monkeypatch.setenv("PAFP8_WAIT_CYCLES", bad)
        db.run()
        o, lse = db.result()
        ro, rl = oracle_on(b)
        assert_close(o, lse, ro, rl, f"PAFP8_WAIT_CYCLES={bad!r}")
