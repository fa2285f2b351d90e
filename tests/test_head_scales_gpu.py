"""Per-head scale tensors (pafp8_run_head_scales) against the oracle with the
same per-head scales, and equal entries against pafp8_run bit for bit, for
decode (split and unsplit rows, fp8 and 2-byte caches, fp8 query) and
prefill (bf16 and fp8 query)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from common import oracle_on
from gpu_common import DeviceBatch, assert_close
from paged_attention_fp8_gb300.workloads import make_batch

pytestmark = pytest.mark.gpu


def _scales(b, seed, equal=False):
    rng = np.random.default_rng(seed)
    hq, hkv = b.num_qo_heads, b.num_kv_heads
    f = (lambda n: np.ones(n)) if equal else (lambda n: rng.uniform(0.4, 2.5, n))
    qs = (f(hq) * b.q_scale).astype(np.float32) if b.q_dtype in ("e4m3fn", "e5m2") else None
    return qs, (f(hkv) * b.k_scale).astype(np.float32), (f(hkv) * b.v_scale).astype(np.float32)


def _run(db, qs, ks, vs):
    dev = db.device
    t = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    db.plan.run_head_scales(db.q, db.k, db.v, db.kv_indices, db.o, db.lse, db.ws, q_scales=t(qs),
                            k_scales=t(ks), v_scales=t(vs))
    return db.result()


CASES = [
    ("decode", dict(kv_lens=[1, 40, 300, 3000], q_dtype="bf16", kv_dtype="e4m3fn"), dict(num_ctas=20)),
    ("decode", dict(kv_lens=[77, 2500], q_dtype="e4m3fn", kv_dtype="e4m3fn"), dict(num_ctas=16)),
    ("decode", dict(kv_lens=[5, 1200], q_dtype="f16", kv_dtype="e5m2"), dict(disable_split_kv=True)),
    ("decode", dict(kv_lens=[33, 900], q_dtype="bf16", kv_dtype="bf16"), dict(num_ctas=8)),
    ("prefill", dict(kv_lens=[300, 129], qo_lens=[200, 129], q_dtype="bf16", kv_dtype="e4m3fn"), dict(num_ctas=5)),
    ("prefill", dict(kv_lens=[260, 64], qo_lens=[260, 30], q_dtype="e4m3fn", kv_dtype="e4m3fn"), dict(num_ctas=5)),
]


@pytest.mark.parametrize("mode,bk,pk", CASES)
def test_per_head_scales_match_the_oracle(cuda_device, mode, bk, pk):
    b = make_batch(bk["kv_lens"], bk.get("qo_lens"), num_qo_heads=16, num_kv_heads=4, q_dtype=bk["q_dtype"],
                   kv_dtype=bk["kv_dtype"], seed=83 + len(bk["kv_lens"]), pool_pages=400)
    db = DeviceBatch(b, cuda_device, **pk)
    qs, ks, vs = _scales(b, 1)
    o, lse = _run(db, qs, ks, vs)
    ro, rl = oracle_on(b, q_scale=qs if qs is not None else b.q_scale, k_scale=ks, v_scale=vs)
    assert_close(o, lse, ro, rl, f"per-head scales {mode} {bk['q_dtype']}/{bk['kv_dtype']}")
    # equal entries: pafp8_run's result bit for bit
    qe, ke, ve = _scales(b, 1, equal=True)
    o2, l2 = _run(db, qe, ke, ve)
    db.run()
    o3, l3 = db.result()
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)
