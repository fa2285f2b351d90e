"""Prefill and decode over one page pool in one call (pafp8_run_pod): each
phase against the oracle, and bit for bit against pafp8_run of the same plan
alone, for SM splits that fit side by side and one that does not."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_attention_fp8_gb300 as pa
from common import oracle_on
from gpu_common import DeviceBatch, assert_close
from paged_attention_fp8_gb300.workloads import make_batch, pod_batch, pod_workload, with_layout

pytestmark = pytest.mark.gpu


def _sms(dev):
    return torch.cuda.get_device_properties(dev).multi_processor_count


class Pod:
    """Device copies of a PodBatch: one cache, a DeviceBatch per phase."""

    def __init__(self, pb, dev, *, prefill_ctas, decode_ctas):
        self.pb = pb
        self.pre = DeviceBatch(pb.prefill, dev, num_ctas=prefill_ctas)
        self.dec = DeviceBatch(pb.decode, dev, num_ctas=decode_ctas)
        self.dec.k, self.dec.v = self.pre.k, self.pre.v  # the one pool

    def run_pod(self):
        b = self.pb.prefill
        pa.pafp8_run_pod(self.pre.plan.handle, self.pre.q, self.pre.kv_indices, self.pre.o, self.pre.lse,
                         self.pre.ws, self.dec.plan.handle, self.dec.q, self.dec.kv_indices, self.dec.o,
                         self.dec.lse, self.dec.ws, self.pre.k, self.pre.v, q_scale=b.q_scale,
                         k_scale=b.k_scale, v_scale=b.v_scale)

    def results(self):
        return self.pre.result(), self.dec.result()


def _check(pod, what, rows=None):
    (po, pl), (do, dl) = pod.results()
    # the same plans run alone, one after the other
    pod.pre.o.zero_(), pod.dec.o.zero_()
    pod.pre.run()
    pod.dec.run()
    (so, sl), (to, tl) = pod.results()
    assert np.array_equal(po, so) and np.array_equal(pl, sl), f"{what}: prefill phase differs from pafp8_run"
    assert np.array_equal(do, to) and np.array_equal(dl, tl), f"{what}: decode phase differs from pafp8_run"
    ro, rl = oracle_on(pod.pb.decode)
    assert_close(do, dl, ro, rl, f"{what}: decode phase")
    if rows is None:
        ro, rl = oracle_on(pod.pb.prefill)
        assert_close(po, pl, ro, rl, f"{what}: prefill phase")
    else:
        r, h = rows
        ro, rl = oracle_on(pod.pb.prefill, rows=r, heads=h)
        assert_close(po[r, h], pl[r, h], ro, rl, f"{what}: prefill phase (sampled)")


@pytest.mark.parametrize("decode_ctas", [8, 24])
def test_pod_scaled_down_side_by_side(cuda_device, decode_ctas):
    pod = Pod(pod_workload(10, scale_down=8), cuda_device, prefill_ctas=_sms(cuda_device) - decode_ctas,
              decode_ctas=decode_ctas)
    pod.run_pod()
    _check(pod, f"POD / 8, {decode_ctas} decode CTAs")


def test_pod_oversubscribed_split(cuda_device):
    """Both grids as wide as the GPU: the later CTAs wait for SMs; same results."""
    n = _sms(cuda_device)
    pod = Pod(pod_workload(10, scale_down=8), cuda_device, prefill_ctas=n, decode_ctas=n)
    pod.run_pod()
    _check(pod, "POD / 8 oversubscribed")


def test_pod_ragged_edges(cuda_device):
    """Decode requests with no KV and one token, prefill tails of one row."""
    pre = make_batch([1, 17, 130, 300], [1, 17, 3, 129], num_qo_heads=16, num_kv_heads=4, seed=71,
                     pool_pages=40)
    dec = make_batch([0, 1, 15, 16, 17, 999], num_qo_heads=16, num_kv_heads=4, seed=72, pool_pages=90)
    pod = Pod(pod_batch(pre, dec), cuda_device, prefill_ctas=5, decode_ctas=3)
    pod.run_pod()
    _check(pod, "POD ragged edges")


def test_pod_full_size_sampled(cuda_device):
    """The bench's POD workload and split: decode in full, prefill on sampled rows."""
    pb = pod_workload(10)
    n = _sms(cuda_device)
    pod = Pod(pb, cuda_device, prefill_ctas=n - 16, decode_ctas=16)
    pod.run_pod()
    g = np.random.default_rng(10)
    b = pb.prefill
    rows = np.concatenate([g.integers(0, b.nnz_qo, 120), b.qo_indptr[1:].numpy() - 1])
    heads = np.concatenate([g.integers(0, b.num_qo_heads, 120), np.full(b.batch, b.num_qo_heads - 1)])
    _check(pod, "POD full size", rows=(rows, heads))


def test_pod_replays_from_a_cuda_graph(cuda_device):
    """The fork and join are stream events, so a POD call captures into a
    graph (after a first call outside capture has made the side stream)."""
    n = _sms(cuda_device)
    pod = Pod(pod_workload(10, scale_down=8), cuda_device, prefill_ctas=n - 16, decode_ctas=16)
    pod.run_pod()
    (po, pl), (do, dl) = pod.results()
    pod.pre.o.zero_(), pod.dec.o.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pod.run_pod()
    g.replay()
    torch.cuda.synchronize()
    (go, gl), (eo, el) = pod.results()
    assert np.array_equal(po, go) and np.array_equal(pl, gl)
    assert np.array_equal(do, eo) and np.array_equal(dl, el)


@pytest.mark.parametrize("variant", ["head64", "hnd_page32", "fp8_query_head64"])
def test_pod_shapes(cuda_device, variant):
    """POD over caches of head_dim 64 and of head-major 32-token pages: each
    phase as alone and against the oracle."""
    d = 64 if "head64" in variant else 128
    P = 32 if variant == "hnd_page32" else 16
    q = "e4m3fn" if variant.startswith("fp8") else "bf16"
    pre = make_batch([60, 300, 129], [60, 200, 1], num_qo_heads=16, num_kv_heads=4, head_dim=d, page_size=P,
                     q_dtype=q, seed=211, pool_pages=1000 // P)
    dec = make_batch([0, 1, 31, 33, 700, 2100], num_qo_heads=16, num_kv_heads=4, head_dim=d, page_size=P,
                     q_dtype=q, seed=212, pool_pages=3200 // P)
    if variant == "hnd_page32":
        pre, dec = with_layout(pre, "HND"), with_layout(dec, "HND")
    pod = Pod(pod_batch(pre, dec), cuda_device, prefill_ctas=_sms(cuda_device) - 12, decode_ctas=12)
    pod.run_pod()
    _check(pod, f"POD {variant}")
