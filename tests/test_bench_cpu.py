"""Host-side arithmetic of bench.py (no GPU).

The roofline fractions the benchmark reports rest on two counts: causal
(t, s) pairs (indexer work) and selected pairs (attention work).  They are
checked here against brute-force enumeration and against the figures for
the long-prefill workload (L = 32768, index_topk = 2048).  The DRAM traffic
figure must be reported only while the attention source matches the source
the counters were taken on.
"""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_attention_long_gemm_b300.synth import CONFIGS  # noqa: E402


@pytest.mark.parametrize("lens,k", [([5, 3], 2), ([1], 4), ([7, 1, 9], 3), ([64, 65], 64)])
def test_work_counts_match_enumeration(lens, k):
    causal = selected = 0
    for L in lens:
        for t in range(L):
            cand = [s for s in range(L) if s <= t]
            causal += len(cand)
            selected += min(k, len(cand))
    assert bench._work_counts(lens, k) == (causal, selected)


def test_work_counts_long_prefill():
    causal, selected = bench._work_counts([32768], 2048)
    assert causal == 32768 * 32769 // 2 == 536_887_296
    # rows t < 2048 keep all t+1 candidates, the other 30720 rows keep 2048
    assert selected == 2048 * 2049 // 2 + 30720 * 2048 == 65_012_736


def _fake_root(tmp_path, source, recorded_sha):
    csrc = tmp_path / "sparse_attention_long_gemm_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "attn_tc.cuh").write_bytes(source)
    (tmp_path / "profiles").mkdir()
    rec = {"attn_tc_kernel_long": {"bytes_per_launch": 123456, "source_sha1": recorded_sha, "how": "test"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    return str(tmp_path)


def test_attn_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    src = b"// kernel source\n"
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, src, hashlib.sha1(src).hexdigest()))
    assert bench._attn_traffic(CONFIGS["long"]) == 123456
    assert bench._attn_traffic(CONFIGS["v32"]) is None          # only the long-prefill launch is scaled


def test_attn_traffic_null_after_a_source_change(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, b"// changed\n", hashlib.sha1(b"// old\n").hexdigest()))
    assert bench._attn_traffic(CONFIGS["long"]) is None



def test_backward_flop_per_pair():
    """The backward's algorithmic work per selected pair, counted term by term: per head the
    logits (2 d_qk), dP (2 d_v), dq (2 d_qk) and dkv (2 d_qk + 2 d_v); per indexer head S, dq_I
    and dk_I (2 D_I each)."""
    v = CONFIGS["v32"]
    per_head = 2 * v.d_qk + 2 * v.d_v + 2 * v.d_qk + (2 * v.d_qk + 2 * v.d_v)
    assert bench.flop_per_pair_attn_bwd(v) == v.n_heads * per_head == 704_512
    assert bench.flop_per_pair_idx_bwd(v) == v.n_idx_heads * 3 * 2 * v.idx_dim == 49_152
    # 2.53 times the forward's attention work per pair (278,528)
    assert bench.flop_per_pair_attn_bwd(v) / bench.flop_per_pair_attn(v) == pytest.approx(2.529, abs=1e-3)
