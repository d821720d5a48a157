"""Host-side pieces of bench.py that set the reported figures (no GPU): the
algorithmic byte counts behind every roofline fraction, the processor lists of
the processors object, and the source hash that ties stored ncu counters to
the kernel they were taken on."""
import numpy as np

import bench


def test_probability_entry_bytes_by_hand():
    # two requests, gamma 3, V = 10, G = 3: request 0 rejects at A = 1, request 1
    # accepts all three drafts (bonus row only)
    V, G = 10, 3
    nacc = np.array([1, 3])
    gam = np.array([3, 3])
    r0 = 4 * 3 + 8 * 2 + 8 * V + 4 + 4 * (G + 1) + 4 + 8 + 8 * (3 - 1)
    r1 = 4 * 3 + 8 * 3 + 4 * V + 4 + 4 * (G + 1) + 4 + 8 + 8 * 0
    assert bench.algorithmic_bytes(nacc, gam, V, G) == r0 + r1


def test_logits_entry_bytes_by_hand():
    # bf16 rows (2 bytes a key): a random request that stops at A = 2 reads
    # target rows 0..2 and draft rows 0..2; one that accepts all 3 reads target
    # rows 0..3 and draft rows 0..2; a greedy request (T = 0) with A = 1 reads
    # target rows 0..1 only
    V, G = 16, 3
    nacc = np.array([2, 3, 1])
    gam = np.array([3, 3, 3])
    temps = np.array([0.8, 1.0, 0.0], np.float32)
    small = lambda A, g: 4 * g + 12 + 4 * (G + 1) + 4 + 8 + 8 * (g - A)
    want = (3 + 3) * V * 2 + small(2, 3) + (4 + 3) * V * 2 + small(3, 3) + 2 * V * 2 + small(1, 3)
    assert bench.logits_algorithmic_bytes(nacc, gam, temps, V, G) == want


def test_processor_lists_layout():
    lists = bench.processor_lists(5, 1000, seed=1, context=7, banned=3, stop=2)
    assert lists["repetition_penalty"].dtype == np.float32 and np.all(lists["repetition_penalty"] == np.float32(1.2))
    for name, n in (("penalty", 7), ("banned", 3), ("stop", 2)):
        cu, ids = lists[f"{name}_cu"], lists[f"{name}_ids"]
        assert cu.dtype == np.int64 and ids.dtype == np.int32
        np.testing.assert_array_equal(cu, np.arange(1, 6) * n)  # inclusive prefix sums
        assert ids.shape == (5 * n,) and ids.min() >= 0 and ids.max() < 1000


def test_source_hash_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    csrc = tmp_path / "speculative_decoding_token_rejection_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    (csrc / "k.cu").write_text("int f(int x) {  // doubled\n  return 2 * x; /* a\n block */ }\n")
    a = bench.kernel_source_hash(["k.cu"])
    (csrc / "k.cu").write_text("// header\nint f(int x) {\n\n    return 2 * x;\n}\n")
    assert bench.kernel_source_hash(["k.cu"]) == a
    (csrc / "k.cu").write_text("int f(int x) { return 3 * x; }\n")
    assert bench.kernel_source_hash(["k.cu"]) != a


def test_stored_traffic_records_resolve():
    """Every committed DRAM traffic record names the hash of the kernel
    sources it was taken on; the bench reads its bytes while that hash matches
    the sources and reports no traffic once it does not."""
    import json
    for name, sources in (("verify_probs_fused_probs", bench.KERNEL_SOURCES),
                          ("verify_logits_fused", bench.LOGITS_KERNEL_SOURCES),
                          ("verify_logits_fused_stream", bench.STREAM_KERNEL_SOURCES),
                          ("draft_sampler_fused_rows", bench.LOGITS_KERNEL_SOURCES),
                          ("draft_sampler_fused_rows_per_row", bench.STREAM_KERNEL_SOURCES),
                          ("ngram_propose_histories", bench.NGRAM_KERNEL_SOURCES)):
        rec = json.loads((bench.ROOT / "profiles" / f"{name}.traffic.json").read_text())
        assert rec["dram_bytes_per_launch"] > 0 and len(rec["kernel_source_sha"]) == 16
        traffic, sha = bench.stored_traffic(name, sources)
        assert sha == rec["kernel_source_sha"]
        if sha == bench.kernel_source_hash(sources):
            assert traffic == rec["dram_bytes_per_launch"]
        else:
            assert traffic is None
