"""The seeded input recipe and the bench's byte accounting (no GPU needed).

The shapes follow the model table of "BitNet Embeddings GGUF Conversion
Implementation", section 1 (Qwen3-shaped 0.6B: hidden 1024, 16 heads of 128,
8 KV heads of 128, FFN 3072; Gemma3-shaped 270M: hidden 640, 4 heads of 256,
one KV head of 256, FFN 2048)."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from bitlinear_rmsnorm_token_gb300 import workloads as wl  # noqa: E402


def _by_name(layer):
    return {p.name: p for p in layer}


def test_layer_tables_chain_like_a_transformer_layer():
    for layer, hidden, attn, kv, ffn in ((wl.QWEN3_0P6B_LAYER, 1024, 16 * 128, 8 * 128, 3072),
                                         (wl.GEMMA3_270M_LAYER, 640, 4 * 256, 1 * 256, 2048)):
        p = _by_name(layer)
        assert [q.name for q in layer] == ["q", "k", "v", "o", "gate", "up", "down"]
        for n in ("q", "k", "v", "gate", "up"):
            assert p[n].K == hidden  # read the hidden state
        assert (p["q"].N, p["k"].N, p["v"].N) == (attn, kv, kv)
        assert (p["o"].K, p["o"].N) == (attn, hidden)
        assert p["gate"].N == p["up"].N == p["down"].K == ffn
        assert p["down"].N == hidden
        for q in layer:
            assert q.K % 128 == 0  # whole I2_S blocks
    assert (wl.QWEN3_0P6B_LAYERS, wl.GEMMA3_270M_LAYERS) == (28, 18)


def test_decode_layer_bytes_of_the_qwen3_layer():
    # per projection: N K / 4 packed bytes + 4 (scale) + x (4 K) + norm_w (4 K) + y (4 N)
    #   q    524288 + 4 + 4096 + 4096 +  8192 = 540676
    #   k    262144 + 4 + 4096 + 4096 +  4096 = 274436, v the same
    #   o    524288 + 4 + 8192 + 8192 +  4096 = 544772
    #   gate 786432 + 4 + 4096 + 4096 + 12288 = 806916, up the same
    #   down 786432 + 4 + 12288 + 12288 + 4096 = 815108
    assert bench.decode_layer_bytes(wl.QWEN3_0P6B_LAYER, 1) == 4063260
    # each extra token adds its x and y rows only
    extra = sum(4 * p.K + 4 * p.N for p in wl.QWEN3_0P6B_LAYER)
    assert bench.decode_layer_bytes(wl.QWEN3_0P6B_LAYER, 2) == 4063260 + extra


def test_draws_are_reproducible_and_distinct():
    a = wl.gen_projection(1, 3, 2, 4, 256, 64)
    b = wl.gen_projection(1, 3, 2, 4, 256, 64)
    for u, v in zip(a, b):
        assert u.dtype == np.float32 and np.array_equal(u, v)
    c = wl.gen_projection(1, 3, 5, 4, 256, 64)  # another projection of the layer
    assert not np.array_equal(a[0], c[0]) and not np.array_equal(a[2], c[2])
    seeds = {wl.seed_for(cfg, layer, proj, t) for cfg in range(2) for layer in range(4) for proj in range(7)
             for t in range(4)}
    assert len(seeds) == 2 * 4 * 7 * 4


def test_outlier_columns():
    M, K = 8, 1024
    base = wl.gen_x(M, K, seed=11)
    x = wl.gen_x(M, K, seed=11, outlier_frac=0.01, outlier_seed=12)
    scaled = np.where(np.any(x != base, axis=0))[0]
    assert len(scaled) == round(0.01 * K)  # 10 of 1024 columns
    assert np.array_equal(x[:, scaled], base[:, scaled] * np.float32(20.0))
    rest = np.setdiff1d(np.arange(K), scaled)
    assert np.array_equal(x[:, rest], base[:, rest])
    # at least one column even when the fraction rounds to none
    y = wl.gen_x(2, 128, seed=3, outlier_frac=0.001)
    assert np.sum(np.any(y != wl.gen_x(2, 128, seed=3), axis=0)) == 1


def test_value_distributions():
    g = wl.gen_norm_w(1 << 16, seed=5)
    assert abs(float(g.mean()) - 1.0) < 0.002 and abs(float(g.std()) - 0.1) < 0.002
    w = wl.gen_latent_w(256, 256, seed=6)
    assert abs(float(w.std()) - 0.02) < 0.0005 and abs(float(w.mean())) < 0.0005
    x = wl.gen_x(64, 1024, seed=7)
    assert abs(float(x.std()) - 1.0) < 0.01 and abs(float(x.mean())) < 0.01
