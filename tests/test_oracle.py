"""Pins of the fp64 oracle against facts fixed outside it: values the pages print,
a hand-worked example, closed forms, special cases that reduce to library
routines, invariants and tiny brute force. CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from mla_latent_kv_13_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def widen(b):
    return synth.bf16_bits_to_f64(b)


# ------------------------------------------------------------------ bf16

@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),                    # tie -> even (1.0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                # tie -> even (1 + 2^-6)
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),       # just above the tie -> up
    (1.0 + 2.0 ** -8 - 2.0 ** -30, 0x3F80),       # just below the tie -> down
    (-2.5, 0xC020),
    (2.0 ** -133, 0x0001),                        # smallest subnormal
    (2.0 ** -134, 0x0000),                        # tie between 0 and 2^-133 -> 0
    (3 * 2.0 ** -134, 0x0002),                    # tie -> even (2^-132)
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),       # largest finite
    ((2 - 2.0 ** -9) * 2.0 ** 127, 0x7F80),       # rounds up past the largest -> inf
    (0.0, 0x0000),
    (-0.0, 0x8000),
])
def test_bf16_rounding_textbook_cases(x, bits):
    assert oracle.f64_to_bf16(x) == bits


def test_bf16_rounding_matches_library_on_fp32_values():
    # For values exactly representable in fp32, rounding fp64 -> bf16 equals the
    # library's fp32 -> bf16 round-to-nearest-even.
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(2000) * np.exp(rng.uniform(-20, 20, 2000))).astype(np.float32)
    ref = bf16(v)
    got = np.array([oracle.f64_to_bf16(float(t)) for t in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(2).standard_normal((5, 64))
    assert np.array_equal(oracle.rope(x, np.zeros(5)), x)


def test_rope_known_rotation():
    # Pair 0 has frequency theta^0 = 1: (1, 0) turns by `pos` radians counter-clockwise.
    # Pair 16 of 64 has frequency theta^(-1/2) = 1/100 at theta = 1e4.
    x = np.zeros((2, 64))
    x[0, 0] = 1.0
    x[1, 32] = 1.0
    y = oracle.rope(x, np.array([3, 100]))
    assert y[0, 0] == pytest.approx(math.cos(3.0), abs=1e-15)
    assert y[0, 1] == pytest.approx(math.sin(3.0), abs=1e-15)
    assert y[1, 32] == pytest.approx(math.cos(1.0), abs=1e-14)
    assert y[1, 33] == pytest.approx(math.sin(1.0), abs=1e-14)
    assert np.count_nonzero(np.abs(y) > 1e-15) == 4


def test_rope_preserves_norm_and_composes():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 64))
    a = np.array([1, 17, 300, 8191])
    b = np.array([5, 2, 1000, 1])
    ya = oracle.rope(x, a)
    np.testing.assert_allclose(np.linalg.norm(ya, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(oracle.rope(ya, b), oracle.rope(x, a + b), atol=1e-10)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    for m, n in [(10, 3), (500, 493), (7, 0)]:
        lhs = float((oracle.rope(q, [m]) @ oracle.rope(k, [n]).T)[0, 0])
        rhs = float((oracle.rope(q, [m - n]) @ k.T)[0, 0])
        assert lhs == pytest.approx(rhs, rel=1e-10, abs=1e-10)


# ------------------------------------------------------- cache-size closed forms

def test_cache_sizes_match_pages():
    g = _golden("cache_sizes.json")
    assert oracle.kv_elements_mha(1, 128, 128) == g["mha_elements_per_token_per_layer_128h_128d"]["value"]
    per_token_bytes = oracle.kv_elements_mla(61, g["latent_dim"]["value"], 64) * 2
    assert round(per_token_bytes / 1024, 1) == g["r1_kv_bytes_per_token_kb"]["value"]
    # the MLA/MHA ratio at 128 heads x 128 dims: 576 / 32768
    assert oracle.kv_elements_mla(1, 512, 64) / oracle.kv_elements_mha(1, 128, 128) == 576 / 32768


# --------------------------------------------------------------- attention

def _tiny_fixture():
    g = _golden("tiny_attention.json")
    bs, dc, dr = g["dims"]["block_size"], g["dims"]["d_c"], g["dims"]["d_rope"]
    nb = 2
    cache = np.full((nb, bs, dc + dr), 0x7FC0, dtype=np.uint16)   # NaN poison everywhere
    bt = np.array([g["block_table"]], dtype=np.int32)
    for j, t in enumerate(g["tokens_logical"]):
        blk = bt[0, j // bs]
        cache[blk, j % bs] = bf16(t["c_kv"] + t["k_rope"])
    q_lat = np.array([[[2 * math.log(2), 2 * (math.log(5) - 1)]]])
    q_rope = np.array([[[2.0, 0.0]]])
    return g, cache, bt, q_lat, q_rope


def test_hand_worked_decode_absorbed():
    g, cache, bt, q_lat, q_rope = _tiny_fixture()
    out, lse, p = oracle.decode_absorbed(q_lat, q_rope, cache, bt, [g["seqlen"]], g["scale"],
                                         want_probs=True)
    np.testing.assert_allclose(out[0, 0], g["expected_out"], rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(g["expected_lse"], abs=1e-15)
    np.testing.assert_allclose(p[:3], g["expected_probs"], atol=1e-15)


def test_hand_worked_decode_expanded():
    g, cache, bt, q_lat, q_rope = _tiny_fixture()
    e = g["expanded"]
    out_v, lse = oracle.decode_expanded(q_lat, q_rope, cache, bt, [g["seqlen"]],
                                        np.array(e["w_uk"]), np.array(e["w_uv"]), g["scale"])
    np.testing.assert_allclose(out_v[0, 0], e["expected_out_v"], atol=1e-15)
    assert lse[0, 0] == pytest.approx(g["expected_lse"], abs=1e-15)


def _random_case(B, H, seqlens, seed, shuffled=True, sigma=1.0):
    w = synth.Workload("t", B, H, tuple(seqlens), None, shuffled)
    return synth.make_attention_inputs(w, seed=seed, sigma=sigma)


def test_one_hot_latents_expose_softmax():
    # c_kv_j = e_j makes o_lat[j] = p_j, which a few lines of plain Python reproduce.
    L, H = 100, 3
    d = _random_case(1, H, [L], seed=5)
    cache = d["kv_cache"].copy()
    bt = d["block_table"]
    for j in range(L):
        row = cache[bt[0, j // 64], j % 64]
        row[:512] = 0
        row[j] = bf16([1.0])[0]
    ql = widen(d["q_lat"])
    qr = widen(d["q_rope"])
    scale = d["scale"]
    out, lse, p = oracle.decode_absorbed(ql, qr, cache, bt, [L], scale, want_probs=True)
    for h in range(H):
        s = []
        for j in range(L):
            kr = widen(cache[bt[0, j // 64], j % 64, 512:])
            s.append(scale * (ql[0, h, j] + sum(qr[0, h, r] * kr[r] for r in range(64))))
        m = max(s)
        den = sum(math.exp(v - m) for v in s)
        pref = [math.exp(v - m) / den for v in s]
        np.testing.assert_allclose(out[0, h, :L], pref, rtol=1e-12, atol=1e-15)
        assert np.all(out[0, h, L:] == 0)
        assert lse[0, h] == pytest.approx(m + math.log(den), rel=1e-13)
    assert math.fsum(p[:L]) == pytest.approx(1.0, abs=1e-14)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 100, 130])
def test_zero_query_gives_mean_and_log_length(L):
    d = _random_case(1, 2, [L], seed=6)
    q0 = np.zeros((1, 2, 512))
    r0 = np.zeros((1, 2, 64))
    out, lse = oracle.decode_absorbed(q0, r0, d["kv_cache"], d["block_table"], [L], d["scale"])
    rows = np.stack([widen(d["kv_cache"][d["block_table"][0, j // 64], j % 64, :512])
                     for j in range(L)])
    np.testing.assert_allclose(out[0, 0], rows.mean(axis=0), rtol=1e-12, atol=1e-14)
    assert lse[0, 1] == pytest.approx(math.log(L), abs=1e-14)


def test_single_token_returns_its_row():
    d = _random_case(1, 4, [1], seed=7)
    ql, qr = widen(d["q_lat"]), widen(d["q_rope"])
    out, lse = oracle.decode_absorbed(ql, qr, d["kv_cache"], d["block_table"], [1], d["scale"])
    row = widen(d["kv_cache"][d["block_table"][0, 0], 0])
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], row[:512])
        s0 = d["scale"] * (float(np.dot(ql[0, h], row[:512])) + float(np.dot(qr[0, h], row[512:])))
        assert lse[0, h] == pytest.approx(s0, rel=1e-12)


def test_empty_sequence():
    d = _random_case(2, 2, [0, 5], seed=8)
    out, lse = oracle.decode_absorbed(widen(d["q_lat"]), widen(d["q_rope"]), d["kv_cache"],
                                      d["block_table"], [0, 5], d["scale"])
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_constant_rows_give_the_row():
    d = _random_case(1, 3, [150], seed=9)
    cache = d["kv_cache"].copy()
    c = bf16(np.random.default_rng(10).standard_normal(576))
    cache[:, :, :] = c
    out, _ = oracle.decode_absorbed(widen(d["q_lat"]), widen(d["q_rope"]), cache,
                                    d["block_table"], [150], d["scale"])
    np.testing.assert_allclose(out[0], np.broadcast_to(widen(c[:512]), (3, 512)), rtol=1e-13)


def test_block_permutation_and_poison_do_not_change_result():
    L = [100, 64]
    d = _random_case(2, 2, L, seed=11, shuffled=False)
    ql, qr = widen(d["q_lat"]), widen(d["q_rope"])
    ref, lref = oracle.decode_absorbed(ql, qr, d["kv_cache"], d["block_table"], L, d["scale"])
    # move every logical block to a new physical slot, poison everything unused
    nb = d["num_blocks"]
    perm = np.random.default_rng(12).permutation(nb + 3)
    big = np.full((nb + 3, 64, 576), 0x7FC0, dtype=np.uint16)
    bt2 = np.full((2, 4), 9999, dtype=np.int32)
    for b in range(2):
        for k in range((L[b] + 63) // 64):
            src = d["block_table"][b, k]
            big[perm[src]] = d["kv_cache"][src]
            bt2[b, k] = perm[src]
    # poison the slots past each sequence's end
    big[bt2[0, 1], 100 - 64:] = 0x7F80
    out, lse = oracle.decode_absorbed(ql, qr, big, bt2, L, d["scale"])
    assert np.array_equal(out, ref) and np.array_equal(lse, lref)


def test_out_of_range_block_is_reported():
    d = _random_case(1, 1, [70], seed=13)
    bt = d["block_table"].copy()
    bt[0, 1] = d["num_blocks"] + 5
    with pytest.raises(oracle.OracleError):
        oracle.decode_absorbed(widen(d["q_lat"]), widen(d["q_rope"]), d["kv_cache"], bt, [70],
                               d["scale"])
    out, lse = oracle.decode_absorbed(widen(d["q_lat"]), widen(d["q_rope"]), d["kv_cache"], bt,
                                      [70], d["scale"], allow_range=True)
    assert np.all(np.isfinite(out))


def test_tiny_brute_force_random():
    # B=1, H=2, L=3 with small dims: a direct evaluation written here in plain Python.
    rng = np.random.default_rng(14)
    dc, dr, L = 4, 2, 3
    cache = bf16(rng.standard_normal((2, 2, dc + dr)))
    bt = np.array([[1, 0]], dtype=np.int32)
    ql = rng.standard_normal((1, 2, dc))
    qr = rng.standard_normal((1, 2, dr))
    out, lse = oracle.decode_absorbed(ql, qr, cache, bt, [L], 0.7)
    rows = [widen(cache[bt[0, j // 2], j % 2]) for j in range(L)]
    for h in range(2):
        s = [0.7 * (sum(ql[0, h, c] * r[c] for c in range(dc)) +
                    sum(qr[0, h, t] * r[dc + t] for t in range(dr))) for r in rows]
        e = [math.exp(v) for v in s]
        o = [sum(e[j] * rows[j][c] for j in range(L)) / sum(e) for c in range(dc)]
        np.testing.assert_allclose(out[0, h], o, rtol=1e-13)
        assert lse[0, h] == pytest.approx(math.log(sum(e)), rel=1e-14)


# ------------------------------------------------------ absorption identity

@pytest.mark.parametrize("B,H,L,seed", [(2, 16, (64, 100), 0), (1, 4, (257,), 3)])
def test_absorbed_equals_expanded(B, H, L, seed):
    """W_UK absorbed into the query and W_UV into the output give exactly the
    expanded multi-head result (fp64, relative 1e-12)."""
    d = _random_case(B, H, L, seed=seed)
    rng = np.random.default_rng(100 + seed)
    q_nope = rng.standard_normal((B, H, 128))
    q_rope = rng.standard_normal((B, H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) * 0.05
    w_uv = rng.standard_normal((H, 128, 512)) * 0.05
    scale = d["scale"]
    out_v, lse_e = oracle.decode_expanded(q_nope, q_rope, d["kv_cache"], d["block_table"], L,
                                          w_uk, w_uv, scale)
    q_lat = np.einsum("hdc,bhd->bhc", w_uk, q_nope)
    o_lat, lse_a = oracle.decode_absorbed(q_lat, q_rope, d["kv_cache"], d["block_table"], L, scale)
    out_a = np.einsum("hdc,bhc->bhd", w_uv, o_lat)
    np.testing.assert_allclose(lse_a, lse_e, rtol=1e-12)
    np.testing.assert_allclose(out_a, out_v, rtol=1e-12, atol=1e-12 * np.abs(out_v).max())


# ------------------------------------------------------------------ combine

def test_combine_of_block_aligned_parts_equals_whole():
    L = 300
    d = _random_case(1, 3, [L], seed=15)
    ql, qr = widen(d["q_lat"]), widen(d["q_rope"])
    bt = d["block_table"]
    full, lfull = oracle.decode_absorbed(ql, qr, d["kv_cache"], bt, [L], d["scale"])
    cuts = [0, 64, 192, 192, 300]   # includes an empty part
    parts, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sub = np.full((1, bt.shape[1]), -1, dtype=np.int32)
        nblk = (b - a + 63) // 64
        sub[0, :nblk] = bt[0, a // 64:a // 64 + nblk]
        o, l = oracle.decode_absorbed(ql, qr, d["kv_cache"], sub, [b - a], d["scale"])
        parts.append(o[:, None])
        lses.append(l[:, None])
    out, lse = oracle.combine(np.concatenate(parts, 1), np.concatenate(lses, 1))
    np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse, lfull, rtol=1e-13)


def test_combine_all_empty():
    out, lse = oracle.combine(np.ones((1, 2, 1, 4)), np.full((1, 2, 1), -np.inf))
    assert np.all(out == 0) and np.isneginf(lse[0, 0])


# ------------------------------------------------------------------- append

def test_append_integer_inputs_exact_and_paged():
    rng = np.random.default_rng(16)
    B, dm = 3, 96
    h = bf16(rng.integers(-2, 3, (B, dm)).astype(np.float32))
    w = bf16(rng.integers(-2, 3, (576, dm)).astype(np.float32))
    bt = np.array([[4, 2], [0, 1], [3, 5]], dtype=np.int32)
    pos = np.array([0, 0, 0], dtype=np.int32)
    cache = np.full((6, 64, 576), 0x1234, dtype=np.uint16)
    before = cache.copy()
    oracle.append_kv(h, w, pos, bt, cache)
    ref = bf16((widen(h) @ widen(w).T).astype(np.float32))   # integers < 256: exact
    for b in range(B):
        assert np.array_equal(cache[bt[b, 0], 0], ref[b])
    mask = np.ones(cache.shape[:2], bool)
    for b in range(B):
        mask[bt[b, 0], 0] = False
    assert np.array_equal(cache[mask], before[mask])


def test_append_real_inputs_within_one_ulp_and_rope_norm():
    rng = np.random.default_rng(17)
    B, dm = 2, 256
    h = bf16(rng.standard_normal((B, dm)))
    w = bf16(rng.standard_normal((576, dm)) * 0.05)
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    c0 = np.zeros((4, 64, 576), dtype=np.uint16)
    oracle.append_kv(h, w, [0, 0], bt, c0)
    x = widen(h) @ widen(w).T
    got0 = np.stack([c0[0, 0], c0[2, 0]]).astype(np.int32)
    ref0 = np.array([[oracle.f64_to_bf16(v) for v in row] for row in x]).astype(np.int32)
    assert np.max(np.abs(got0 - ref0)) <= 1
    c1 = np.zeros_like(c0)
    oracle.append_kv(h, w, [70, 127], bt, c1)
    got1 = np.stack([c1[1, 6], c1[3, 63]])
    assert np.array_equal(got1[:, :512], np.stack([c0[0, 0], c0[2, 0]])[:, :512])
    n0 = np.linalg.norm(x[:, 512:], axis=1)
    n1 = np.linalg.norm(widen(got1[:, 512:]), axis=1)
    np.testing.assert_allclose(n1, n0, rtol=1e-2)


# ---------------------------------------------------------- projections

def _proj_weights(B, dm, ql, H, seed):
    rng = np.random.default_rng(seed)
    s = 0.05
    return dict(
        h=bf16(rng.standard_normal((B, dm))),
        w_dq=bf16(rng.standard_normal((ql, dm)) * s),
        w_uq=bf16(rng.standard_normal((H * 128, ql)) * s),
        w_qr=bf16(rng.standard_normal((H * 64, ql)) * s),
        w_uk=bf16(rng.standard_normal((H, 128, 512)) * s),
        w_uv=bf16(rng.standard_normal((H, 128, 512)) * s),
        w_o=bf16(rng.standard_normal((dm, H * 128)) * s),
    )


def test_absorb_q_matches_matrix_products_at_position_zero():
    B, dm, ql, H = 3, 64, 48, 2
    p = _proj_weights(B, dm, ql, H, 18)
    q_lat, q_rope, q_nope = oracle.absorb_q(p["h"], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"],
                                            np.zeros(B), want_nope=True)
    cq = widen(p["h"]) @ widen(p["w_dq"]).T
    qn = (cq @ widen(p["w_uq"]).T).reshape(B, H, 128)
    qr = (cq @ widen(p["w_qr"]).T).reshape(B, H, 64)
    ql_ref = np.einsum("bhd,hdc->bhc", qn, widen(p["w_uk"]))
    np.testing.assert_allclose(q_nope, qn, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(q_rope, qr, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(q_lat, ql_ref, rtol=1e-11, atol=1e-14)


def test_absorb_q_position_only_moves_rope_part():
    B, dm, ql, H = 2, 64, 32, 2
    p = _proj_weights(B, dm, ql, H, 19)
    a = oracle.absorb_q(p["h"], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"], [0, 0])
    b = oracle.absorb_q(p["h"], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"], [5, 4000])
    assert np.array_equal(a[0], b[0])
    np.testing.assert_allclose(np.linalg.norm(b[1], axis=2), np.linalg.norm(a[1], axis=2),
                               rtol=1e-13)
    assert not np.allclose(a[1], b[1])


def test_absorbed_query_scores_latents_like_expanded_keys():
    # q_lat . c == q_nope . (W_UK c) for any latent c (the absorption on the query side).
    B, dm, ql, H = 2, 64, 32, 3
    p = _proj_weights(B, dm, ql, H, 20)
    q_lat, _, q_nope = oracle.absorb_q(p["h"], p["w_dq"], p["w_uq"], p["w_qr"], p["w_uk"],
                                       [1, 2], want_nope=True)
    c = np.random.default_rng(21).standard_normal(512)
    k = np.einsum("hdc,c->hd", widen(p["w_uk"]), c)
    np.testing.assert_allclose(q_lat @ c, np.einsum("bhd,hd->bh", q_nope, k), rtol=1e-11)


def test_out_absorb_matches_matrix_products():
    B, dm, H = 3, 40, 2
    p = _proj_weights(B, dm, 8, H, 22)
    o_lat = np.random.default_rng(23).standard_normal((B, H, 512))
    y = oracle.out_absorb(o_lat, p["w_uv"], p["w_o"])
    ov = np.einsum("hdc,bhc->bhd", widen(p["w_uv"]), o_lat).reshape(B, H * 128)
    np.testing.assert_allclose(y, ov @ widen(p["w_o"]).T, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- multi-query decode


@pytest.mark.parametrize("L,s_q", [(1, 1), (5, 2), (64, 4), (65, 3), (130, 4)])
def test_multi_query_zero_query_sees_exactly_its_causal_prefix(L, s_q):
    """q = 0 turns every draft token's output into the mean of the rows it sees and its
    lse into ln(count): draft token t sees L - (s_q - 1 - t) rows (closed form)."""
    d = _random_case(1, 2, [L], seed=40)
    q0 = np.zeros((1, s_q, 2, 512))
    r0 = np.zeros((1, s_q, 2, 64))
    out, lse = oracle.decode_absorbed_mq(q0, r0, d["kv_cache"], d["block_table"], [L],
                                         d["scale"])
    rows = np.stack([widen(d["kv_cache"][d["block_table"][0, j // 64], j % 64, :512])
                     for j in range(L)])
    for t in range(s_q):
        n = L - (s_q - 1 - t)
        if n <= 0:
            assert np.all(out[0, t] == 0) and np.all(np.isneginf(lse[0, t]))
            continue
        np.testing.assert_allclose(out[0, t, 1], rows[:n].mean(axis=0), rtol=1e-12, atol=1e-14)
        assert lse[0, t, 0] == pytest.approx(math.log(n), abs=1e-14)


def test_multi_query_draft_tokens_never_see_later_rows():
    """Poisoning the rows after draft token t's visible prefix leaves its result alone and
    changes the later tokens'; the last token sees the whole sequence."""
    B, H, s_q, L = 2, 4, 3, 150
    d = _random_case(B, H, [L, L - 20], seed=41)
    rng = np.random.default_rng(42)
    q = rng.standard_normal((B, s_q, H, 512)) * 0.3
    r = rng.standard_normal((B, s_q, H, 64)) * 0.3
    Ls = [L, L - 20]
    out, lse = oracle.decode_absorbed_mq(q, r, d["kv_cache"], d["block_table"], Ls, d["scale"])
    cache = d["kv_cache"].copy()
    for b in range(B):  # overwrite the last two rows of each sequence
        for j in (Ls[b] - 2, Ls[b] - 1):
            cache[d["block_table"][b, j // 64], j % 64, :] = bf16(rng.standard_normal(576) * 5)
    out2, lse2 = oracle.decode_absorbed_mq(q, r, cache, d["block_table"], Ls, d["scale"])
    np.testing.assert_array_equal(out2[:, 0], out[:, 0])   # sees rows < L - 2
    np.testing.assert_array_equal(lse2[:, 0], lse[:, 0])
    assert not np.allclose(out2[:, 1], out[:, 1])            # sees row L - 2
    assert not np.allclose(out2[:, 2], out[:, 2])
    for b in range(B):  # the last draft token is plain decode over the whole sequence
        o1, l1 = oracle.decode_absorbed(q[b:b + 1, s_q - 1], r[b:b + 1, s_q - 1], d["kv_cache"],
                                        d["block_table"][b:b + 1], [Ls[b]], d["scale"])
        np.testing.assert_array_equal(out[b, s_q - 1], o1[0])
        np.testing.assert_array_equal(lse[b, s_q - 1], l1[0])


# ---------------------------------------------------------------- chunked prefill


@pytest.mark.parametrize("prefix,C", [(0, 5), (70, 3), (128, 2)])
def test_prefill_zero_query_averages_the_projected_prefix(prefix, C):
    """q = 0: query i weighs its prefix + i + 1 visible rows equally, so out_v is W_UV
    applied to their mean latent and lse = ln(prefix + i + 1) (closed form)."""
    L = prefix + C
    d = _random_case(1, 2, [L], seed=50)
    rng = np.random.default_rng(51)
    w_uk = rng.standard_normal((2, 128, 512)) * 0.05
    w_uv = rng.standard_normal((2, 128, 512)) * 0.05
    out, lse = oracle.prefill_expanded(np.zeros((C, 2, 128)), np.zeros((C, 2, 64)),
                                       d["kv_cache"], d["block_table"][0], prefix, w_uk, w_uv,
                                       d["scale"])
    rows = np.stack([widen(d["kv_cache"][d["block_table"][0, j // 64], j % 64, :512])
                     for j in range(L)])
    for i in range(C):
        n = prefix + i + 1
        np.testing.assert_allclose(out[i, 1], w_uv[1] @ rows[:n].mean(axis=0), rtol=1e-11,
                                   atol=1e-13)
        assert lse[i, 0] == pytest.approx(math.log(n), abs=1e-13)


def test_prefill_expanded_equals_absorbed_per_query():
    """Each query of the chunk, expanded (K, V projected per head), equals the absorbed form
    (W_UK folded into the query, W_UV applied to the latent output) over its causal prefix."""
    prefix, C, H = 90, 6, 3
    d = _random_case(1, H, [prefix + C], seed=52)
    rng = np.random.default_rng(53)
    q_nope = rng.standard_normal((C, H, 128))
    q_rope = rng.standard_normal((C, H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) * 0.05
    w_uv = rng.standard_normal((H, 128, 512)) * 0.05
    out, lse = oracle.prefill_expanded(q_nope, q_rope, d["kv_cache"], d["block_table"][0],
                                       prefix, w_uk, w_uv, d["scale"])
    for i in range(C):
        q_lat = np.einsum("hdc,hd->hc", w_uk, q_nope[i])[None]
        o_lat, l_a = oracle.decode_absorbed(q_lat, q_rope[i][None], d["kv_cache"],
                                            d["block_table"], [prefix + i + 1], d["scale"])
        np.testing.assert_allclose(lse[i], l_a[0], rtol=1e-12)
        np.testing.assert_allclose(out[i], np.einsum("hdc,hc->hd", w_uv, o_lat[0]), rtol=1e-10,
                                   atol=1e-12)


def test_prefill_query_never_sees_later_rows():
    prefix, C, H = 40, 4, 2
    d = _random_case(1, H, [prefix + C], seed=54)
    rng = np.random.default_rng(55)
    q_nope = rng.standard_normal((C, H, 128))
    q_rope = rng.standard_normal((C, H, 64))
    w_uk = rng.standard_normal((H, 128, 512)) * 0.05
    w_uv = rng.standard_normal((H, 128, 512)) * 0.05
    bt = d["block_table"][0]
    out, lse = oracle.prefill_expanded(q_nope, q_rope, d["kv_cache"], bt, prefix, w_uk, w_uv,
                                       d["scale"])
    cache = d["kv_cache"].copy()
    j = prefix + C - 1  # the chunk's last row: only the last query sees it
    cache[bt[j // 64], j % 64, :] = bf16(rng.standard_normal(576) * 4)
    out2, lse2 = oracle.prefill_expanded(q_nope, q_rope, cache, bt, prefix, w_uk, w_uv, d["scale"])
    np.testing.assert_array_equal(out2[:C - 1], out[:C - 1])
    np.testing.assert_array_equal(lse2[:C - 1], lse[:C - 1])
    assert not np.allclose(out2[C - 1], out[C - 1])
