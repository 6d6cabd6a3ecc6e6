"""The seeded input generators (CPU side)."""
import numpy as np

from synth import kvgen, workloads


def test_splitmix64_published_sequence():
    # SplitMix64 seeded with 0 (Steele, Lea & Flood 2014; Vigna's reference
    # generator) starts 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4.
    w = kvgen.words(np.uint64(0), np.arange(2))
    assert [int(x) for x in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_irwin_hall_moments_and_determinism():
    x = kvgen.irwin_hall_f32(7, 0, np.arange(400000))
    assert abs(float(x.mean())) < 0.01
    assert abs(float(x.var()) - 1.0) < 0.01
    assert np.all(np.abs(x) <= 6.0)
    assert np.array_equal(x, kvgen.irwin_hall_f32(7, 0, np.arange(400000)))
    assert not np.array_equal(x[:1000], kvgen.irwin_hall_f32(7, 1, np.arange(1000)))
    # exact multiples of 2^-16
    assert np.all((x.astype(np.float64) * 65536.0) % 1.0 == 0.0)


def test_kv_elements_chunking_consistent():
    a = kvgen.kv_elements(3, 1, 1000, 5000, "bf16", chunk=777)
    b = kvgen.kv_elements(3, 1, 1000, 5000, "bf16")
    assert np.array_equal(a, b)
    c = kvgen.kv_elements(3, 1, 3000, 10, "bf16")
    assert np.array_equal(b[2000:2010], c)


def test_workload_shapes():
    wl = workloads.get("tiny")
    s = wl.spec
    assert wl.lengths.min() >= 4 and wl.lengths.max() <= 16 and len(wl.lengths) == 64
    assert np.allclose(np.linalg.norm(wl.emb.astype(np.float64), axis=1), 1.0, atol=1e-6)
    assert sorted(wl.block_table[0]) == list(range(32))
    K = wl.fact_kv(3, kvgen.STREAM_K)
    assert K.shape == (wl.lengths[3], s.num_layers, s.num_kv_heads, s.head_dim)
    wl2 = workloads.get("qwen25_7b_100u")
    assert wl2.block_table.shape[0] == 100
    used = wl2.block_table[wl2.block_table > 0]
    assert len(np.unique(used)) == len(used)             # distinct physical blocks
    assert wl2.num_blocks == 1 + len(used)
    assert np.all(wl2.users == np.arange(100))
