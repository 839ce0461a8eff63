"""The seeded input generator: determinism, slice addressability, workload recipes."""
import numpy as np

import synth
from oracle import widen_bf16


def test_same_seed_same_bits_and_slices_regenerate():
    a = synth.normal_bf16(7, synth.stream_id(synth.T_K, 3, 2), 10000)
    b = synth.normal_bf16(7, synth.stream_id(synth.T_K, 3, 2), 10000)
    assert np.array_equal(a, b)
    c = synth.normal_bf16(7, synth.stream_id(synth.T_K, 3, 2), 500, start=1234)
    assert np.array_equal(a[1234:1734], c)
    d = synth.normal_bf16(8, synth.stream_id(synth.T_K, 3, 2), 10000)
    assert not np.array_equal(a, d)


def test_normal_statistics():
    x = widen_bf16(synth.normal_bf16(1, 2, 400000))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert x.min() >= -6.0 and x.max() <= 6.0


def test_unit_vector_and_heavy_keys():
    w = synth.WORKLOADS["llama8b"]
    u = w.direction(0, 0).astype(np.float64)
    assert abs(np.linalg.norm(u) - 1.0) < 1e-6
    n = 4096
    kind = w.key_kinds(0, 0, n)
    assert (kind == 1).sum() == int(np.floor(0.02 * n)) and (kind == 2).sum() == 0
    K = widen_bf16(synth.keys_bf16(w.seed, synth.stream_id(synth.T_K, 0, 0), 0, n, w.Hkv, w.d, kind, u))
    proj = K @ u                                            # [n][Hkv]
    assert proj[kind == 1].mean() > 2.5 and abs(proj[kind == 0].mean()) < 0.1


def test_prefix_slices_match_whole_sequence():
    w = synth.scaled(synth.WORKLOADS["long70b"], n=2000)
    full = w.prefix_k(0, 0)
    part = w.prefix_k(0, 0, pos0=700, npos=300)
    assert np.array_equal(full[700:1000], part)
    kind = w.key_kinds(0, 0, 2000)
    assert (kind[:16] == 2).all() and (kind == 1).sum() == 20
    sink = widen_bf16(full[:16])
    assert np.allclose(sink[0], sink[5])                    # sinks are exactly 4u


def test_ragged_lengths_and_layout():
    w = synth.WORKLOADS["loop32"]
    n = w.lengths()
    assert n.shape == (8,) and n.min() >= 4096 and n.max() <= 65536
    assert np.array_equal(n, w.lengths(5))                  # same lengths for every layer
    off, slots = w.slot_layout()
    assert off[0] == 0 and np.all(np.diff(off) >= n[:-1] + w.R) and slots >= off[-1] + n[-1] + w.R
    assert np.all(off % 16 == 0)


def test_layer_pool_shapes():
    w = synth.scaled(synth.WORKLOADS["batched"], B=2, n=100)
    p = w.layer_pool(0)
    assert p["K"].shape == (p["slots"], 8, 128)
    assert p["q_verify"].shape == (2, 8, 32, 128)
    assert p["q_draft"].shape == (7, 2, 32, 128)
    o = int(p["seq_offset"][1])
    assert np.array_equal(p["K"][o:o + 100], w.prefix_k(0, 1))
    assert not p["K"][100:o].any()                          # reserved slots start empty
