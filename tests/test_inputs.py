"""The seeded input generator (shared by both sides) and the page figures."""
import json
import math
import os

import numpy as np

import oracle.flce_oracle as O
import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


def _splitmix_reference(x, count):
    """SplitMix64 written out with Python integers (Vigna's published next())."""
    out, m = [], (1 << 64) - 1
    for _ in range(count):
        x = (x + 0x9E3779B97F4A7C15) & m
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 from state 0, as published with the generator.
    z = np.empty(4, dtype=np.uint64)
    si._splitmix_into(z, np.empty_like(z), np.uint64(0), 0)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                   0x06C45D188009454F, 0xF88BB8A8724C81EC]
    key = si.stream_key(1004, 2)
    z = np.empty(1000, dtype=np.uint64)
    si._splitmix_into(z, np.empty_like(z), key, 0)
    assert [int(v) for v in z] == _splitmix_reference(int(key), 1000)


def test_blocks_and_offsets_agree():
    a = si._normals_block(3, 1, 5, 11)
    b = si._normals_block(3, 1, 0, 20)[5:16]
    assert np.array_equal(a, b)
    big = si.normal_bf16(9, 2, (3 * si._CHUNK + 17,), 1.0)  # spans several threaded blocks
    assert np.array_equal(big[-17:], si.normal_bf16(9, 2, (3 * si._CHUNK + 17,), 1.0)[-17:])
    assert np.array_equal(big[:1000], si.normal_bf16(9, 2, (1000,), 1.0))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-3], dtype=np.float32)
    bits = si.float32_to_bf16_bits(x)
    back = si.bf16_to_float32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                      # tie -> even (mantissa 0)
    assert back[2] == 1.0 + 4 * 2 ** -8        # tie -> even (rounds up)
    assert back[3] == 1.0
    assert back[4] == -2.5
    assert abs(back[5] - 3.0e-3) <= 2 ** -8 * 3.0e-3  # unit roundoff of an 8-bit significand


def test_distributions():
    w = si.bf16_to_float32(si.normal_bf16(1004, 2, (1 << 20,), 0.02)).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.0005 and abs(w.mean()) < 1e-4
    inp = si.make_flce_inputs(2000, 8, 1000, 5, ignore_frac=0.05)
    assert int((inp.target == -100).sum()) == 100
    ok = inp.target[inp.target != -100]
    assert ok.min() >= 0 and ok.max() < 1000
    z = si.zipf_targets(1, 4, 200000, 1000, 1.1)
    counts = np.bincount(z, minlength=1000)
    # P(k) ~ k^-1.1: the ratio of the first two frequencies is 2^1.1
    assert abs(counts[0] / counts[1] - 2 ** 1.1) < 0.1


def test_page_figures_pin_byte_accounting():
    g = json.load(open(GOLDEN))
    e = g["logits_example"]
    n_bytes = O.full_logits_bytes(e["batch"] * e["seq_len"], e["vocab"], e["bytes_per_logit"])
    assert round(n_bytes / 1e9, 1) == e["printed_gb"]
    p = g["l20_memory_profile"]
    assert round(p["torch_peak_bytes"] / 2 ** 20, 2) == p["torch_peak_mib"]
    assert round(p["liger_peak_bytes"] / 2 ** 20, 2) == p["liger_peak_mib"]
    one = O.full_logits_bytes(p["tokens_per_rank"], p["local_vocab"], p["bytes_per_logit"])
    saved = p["torch_peak_bytes"] - p["liger_peak_bytes"]
    # the fused CE saves three logits-sized bf16 buffers
    assert abs(saved / one - 3.0) < 1e-3
    r = g["rtx5090_ce_op"]
    for row in r["rows"]:
        one = O.full_logits_bytes(row["tokens"], r["local_vocab"], r["bytes_per_logit"]) / 2 ** 30
        assert abs((row["torch_gib"] - row["liger_gib"]) / one - 3.0) < 0.01
    assert math.isclose(r["rows"][1]["tokens"] / r["rows"][0]["tokens"], 2.0)
