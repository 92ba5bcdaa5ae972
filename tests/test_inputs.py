"""The seeded input recipe (sdm_inputs) holds the properties the workloads state, and the
benchmark's algorithmic byte count (the roofline's numerator) matches a count by sets (no GPU)."""

import os
import sys

import numpy as np
import pytest
import torch

import sdm_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def small(i, **kw):
    base = si.WORKLOADS[i]
    size = dict(P=min(base.P, 3), T=min(base.T, 300), S=min(base.S, 4096))
    size.update(kw)
    return base.replace(**size)


@pytest.mark.parametrize("i", [0, 1, 2, 3, 4])
def test_recipe_properties(i):
    wl = small(i)
    x = si.generate(wl)
    P, T, W, R, S = wl.P, wl.T, wl.W, wl.R, wl.S
    valid = x["valid"]
    assert valid.shape == (P,) and valid.dtype == np.int32
    if wl.ragged:
        assert np.all((valid >= T // 2) & (valid <= T))
    else:
        assert np.all(valid == T)
    for name, width in (("write_slots", W), ("read_slots", R)):
        sl = x[name]
        assert sl.shape == (P, T, width) and sl.dtype == np.int32
        for p in range(P):
            live = sl[p, :valid[p]]
            assert live.min() >= 0 and live.max() < S
            srt = np.sort(live, axis=1)
            assert np.all(srt[:, 1:] != srt[:, :-1]), "slots repeat within a token"
    f = lambda k: si.stored_to_f64(x[k], wl.dtype)  # noqa: E731
    for name in ("write_w", "read_w"):
        w = f(name)
        for p in range(P):
            live = w[p, :valid[p]]
            assert np.all(live > 0)
            # softmax weights: each token's sum is 1 up to the stored dtype's rounding
            tol = 1e-5 if wl.dtype == "f32" else 2e-2
            assert np.abs(live.sum(axis=-1) - 1).max() <= tol
    g, beta = x["log_decay"], x["beta"]
    for p in range(P):
        assert np.all(g[p, :valid[p]] < 0)                  # -0.1 softplus(.) < 0
        assert np.all((beta[p, :valid[p]] > 0) & (beta[p, :valid[p]] < 1))
        # padding inputs are staged as zeros
        for name in ("write_slots", "read_slots", "write_w", "read_w", "log_decay", "v"):
            assert not np.any(x[name][p, valid[p]:]), (name, p)
        assert not np.any(beta[p, valid[p]:])


def test_bf16_storage_is_round_to_nearest_even():
    wl = small(1)
    x = si.generate(wl)
    v = si.stored_to_f64(x["v"], "bf16").astype(np.float32)
    # every stored value is a bfloat16 value (its low 16 bits are zero) ...
    assert not np.any(v.view(np.uint32) & 0xFFFF)
    # ... and the generator's rounding agrees with torch's on arbitrary float32 values
    r = np.random.default_rng(3).standard_normal(10000).astype(np.float32)
    ours = si.bf16_bits_to_f32(si.f32_to_bf16_bits(r))
    ref = torch.from_numpy(r).bfloat16().float().numpy()
    np.testing.assert_array_equal(ours, ref)


def test_zipf_ranks_are_heavy_headed_and_mix_is_half_and_half():
    rng = np.random.default_rng(5)
    z = si.draw_slots(rng, 20000, 16, 65536, "zipf1.1")
    counts = np.bincount(z.ravel(), minlength=8)[:8]
    assert np.all(np.diff(counts) < 0), counts             # slot 0 is the hottest, then 1, ...
    m = si.draw_slots(np.random.default_rng(6), 4000, 64, 1 << 20, "mix")
    head, tail = m[:, :32], m[:, 32:]
    # the Zipf half concentrates on low ids, the uniform half spreads over [0, S)
    assert np.median(head) < 1000 and np.median(tail) > (1 << 18)


def test_generation_is_deterministic():
    wl = small(2)
    a, b = si.generate(wl), si.generate(wl)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    c = si.generate(wl, seed=wl.seed + 1)
    assert not np.array_equal(a["write_slots"], c["write_slots"])


@pytest.mark.parametrize("i", [1, 2, 4])
def test_algorithmic_bytes_by_sets(i):
    """Per chunk: every distinct row touched (writes and reads of the valid tokens) read once,
    every distinct written row written once."""
    sys.path.insert(0, ROOT)
    import bench

    wl = small(i, T=200)
    x = si.generate(wl)
    got = bench.algorithmic_bytes(wl, x)
    row = wl.D * (4 if wl.dtype == "f32" else 2)
    g_rows = dw_rows = 0
    for p in range(wl.P):
        for c0 in range(0, int(x["valid"][p]), wl.C):
            c1 = min(int(x["valid"][p]), c0 + wl.C)
            uw = set(x["write_slots"][p, c0:c1].ravel().tolist())
            ur = set(x["read_slots"][p, c0:c1].ravel().tolist())
            g_rows += len(uw | ur)
            dw_rows += len(uw)
    assert got == {"gather": g_rows * row, "dw": 2 * dw_rows * row,
                   "phase2": (g_rows + dw_rows) * row}


@pytest.mark.parametrize("i", [1, 2, 4])
def test_gram_pairs_by_slot_lists(i):
    """The Phase-1 roofline's unit: per chunk, the pairs of writes of one slot at tokens u < t
    (terms of A) and the pairs (read of slot s at token t, write of s at u <= t) (terms of QK),
    counted here slot by slot from lists of tokens."""
    sys.path.insert(0, ROOT)
    import bench

    wl = small(i, T=300)
    x = si.generate(wl)
    want = 0
    for p in range(wl.P):
        for c0 in range(0, int(x["valid"][p]), wl.C):
            c1 = min(int(x["valid"][p]), c0 + wl.C)
            wtok = {}
            for t in range(c1 - c0):
                for s in x["write_slots"][p, c0 + t].tolist():
                    wtok.setdefault(s, []).append(t)
            for toks in wtok.values():
                want += sum(1 for a in range(len(toks)) for b in range(a + 1, len(toks))
                            if toks[a] < toks[b])
            for t in range(c1 - c0):
                for s in x["read_slots"][p, c0 + t].tolist():
                    want += sum(1 for u in wtok.get(s, ()) if u <= t)
    assert bench.gram_pairs(wl, x) == want


def test_traffic_record_follows_its_sources(tmp_path, monkeypatch):
    """A recorded DRAM byte count is reported for its own kernel family and workload only, and
    only while the sources it names are unchanged."""
    sys.path.insert(0, ROOT)
    import hashlib
    import json

    import bench

    src = tmp_path / "sparse_addressed_delta_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel one\n")
    digest = hashlib.sha256(b"kernel one\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.json").write_text(json.dumps({"dw": [{
        "kernel": "k_dw", "workload": "w_a", "sources": ["k.cu"], "sources_sha256_16": digest,
        "dram_bytes_per_launch": 1234, "capture": "test"}]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("dw", "w_a") == 1234.0
    assert bench.traffic_record("dw", "w_b") is None
    assert bench.traffic_record("gather", "w_a") is None
    (src / "k.cu").write_text("kernel two\n")
    assert bench.traffic_record("dw", "w_a") is None
