"""The byte and FLOP model behind bench.py's roofline numbers, on the CPU.

* ChunkAttention, Knowl 9: plain decode attention (one query row per KV head,
  every sequence reading its own K/V, fp16) has an arithmetic intensity of
  about 0.99 FLOP per byte -- tests/golden/intensity.txt.  The bench's FLOP
  count (4d per query row and key) over its byte count (K/V + q + out) must
  land there; counting only q.k, or K without V, or 4-byte elements, would
  miss it by a factor of two.
* The chunked-prefill FLOPs are brute-forced row by row.
* The split of a step's bytes between the two phases adds up to the step.
"""
import os

import pytest

import bench
from prefix_shared_kv_tree_gb300 import workloads as W


def _golden_intensity():
    path = os.path.join(os.path.dirname(__file__), "golden", "intensity.txt")
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            value, tol = (float(x) for x in line.split())
            return value, tol
    raise AssertionError("no value in intensity.txt")


@pytest.mark.parametrize("name", ["noshare", "share1k", "batch16", "div_s1024_c256", "gen_d64_c64"])
def test_plain_decode_intensity_matches_knowl9(name):
    value, tol = _golden_intensity()
    spec = W.SPECS[name]
    assert spec.group == 1 and spec.dtype == "f16"
    assert abs(bench.plain_decode_intensity(spec) - value) <= tol


def test_intensity_pin_catches_plausible_mistakes():
    value, tol = _golden_intensity()
    spec = W.SPECS["noshare"]
    good = bench.plain_decode_intensity(spec)
    for wrong in (good / 2, good * 2):  # q.k only; K without V (or 4-byte elements)
        assert abs(wrong - value) > tol


def test_prefill_flops_brute_force():
    hq, d = 32, 128
    for p0, w in ((2048, 512), (2560, 512), (3072, 113), (0, 1), (5, 7)):
        brute = sum(4 * d * hq * (p0 + t + 1) for t in range(w))
        assert bench.prefill_flops(p0, w, hq, d) == brute
    # the GQA tree's prompt: 1137 rows after a 2048-token root, as 512 / 512 / 113
    total = sum(bench.prefill_flops(2048 + o, w, 32, 128) for o, w in ((0, 512), (512, 512), (1024, 113)))
    assert total == bench.prefill_flops(2048, 1137, 32, 128)
    assert abs(total / 1e9 - 48.75) < 0.01


@pytest.mark.parametrize("name", ["share1k", "share4k", "noshare", "gqa_tree", "batch96", "tiny"])
def test_phase_bytes_add_up(name):
    spec = W.SPECS[name]
    qo = bench.qo_bytes(spec)
    assert bench.shared_bytes(spec) + bench.private_bytes(spec) == spec.unique_kv_bytes() + 2 * qo
    assert bench.step_bytes(spec) == spec.unique_kv_bytes() + 2 * qo
    if name == "share1k":  # the 1024-token root is the only shared segment: 16 KiB per token
        assert bench.shared_bytes(spec) == 1024 * 16384 + qo
    if name == "noshare":
        assert bench.shared_bytes(spec) == qo


def test_distribution():
    d = bench.distribution([0.001 * x for x in range(1, 101)])  # 1 .. 100 us
    assert d["n"] == 100 and d["median"] == pytest.approx(50.5) and d["mean"] == pytest.approx(50.5)
    assert d["p10"] == pytest.approx(11.0) and d["p90"] == pytest.approx(90.0)


def test_source_digest_ignores_comments_only():
    """A kernel summary's DRAM counters stay attached to the code they were
    taken on: comments and layout do not change the digest, code does."""
    a = 'int f(int x) { // twice\n  return 2 * x; /* no overflow\n here */ }\nconst char* s = "//kept";\n'
    b = 'int f(int x) {\n\n  return 2 * x;   }\n  const char* s = "//kept";  // a literal\n'
    c = 'int f(int x) { return 3 * x; }\nconst char* s = "//kept";\n'
    d = 'int f(int x) { return 2 * x; }\nconst char* s = "kept";\n'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    assert bench.strip_comments(a) != bench.strip_comments(d)
