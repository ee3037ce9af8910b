"""Pins for the fp64 oracle: each checks it against something other than itself.

CPU only.  The pins are a hand-worked example, a textbook stable sort and
numpy's stable argsort, brute force over permutations, dense numpy matmuls
for one-adapter batches (a library routine), associativity of shrink then
expand, exact small-integer arithmetic, permutation invariance and the
special cases (scale 0, zero weights, zero base, one-hot rows).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from gathered_rank_gemm_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def bits(a):
    return W.f32_to_bf16_bits(np.asarray(a, np.float32))


def val(b):
    return oracle.bf16_bits_to_f64(b)


def key_of(m, n, L):
    k = np.asarray(m[:n], np.int64).copy()
    k[(k < 0) | (k >= L)] = L
    return k


# ---------------------------------------------------------------- metadata

def test_metadata_worked_example():
    g = json.load(open(GOLDEN))
    for case in g["metadata"]:
        m = np.array(case["token_lora_mapping"], np.int32)
        s, c, st, status = oracle.prepare_metadata(m, case["num_tokens"], case["max_loras"])
        assert s.tolist() == case["sorted_token_ids"]
        assert c.tolist() == case["num_tokens_per_lora"]
        assert st.tolist() == case["lora_token_start_loc"]
        assert status == case["status"]


def _check_against_argsort(m, n, L):
    s, c, st, _ = oracle.prepare_metadata(m, n, L)
    key = key_of(m, n, L)
    expect = np.argsort(key, kind="stable")
    assert np.array_equal(s[:n], expect)
    assert np.all(s[n:] == -1)
    assert np.array_equal(c, np.bincount(key, minlength=L + 1))
    assert np.array_equal(st, np.concatenate([[0], np.cumsum(np.bincount(key, minlength=L + 1))]))


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_metadata_matches_numpy_stable_argsort_on_every_workload(name):
    shape = W.CONFIGS[name]
    m = W.make_mapping(shape, np.random.default_rng(1000 + shape.index))
    _check_against_argsort(m, shape.num_tokens, shape.max_loras)


def test_metadata_matches_textbook_insertion_sort():
    # a stable sort written the other way round: insertion sort on (key) pairs
    rng = np.random.default_rng(7)
    for _ in range(50):
        L = int(rng.integers(1, 9))
        T = int(rng.integers(0, 70))
        n = int(rng.integers(0, T + 1))
        m = rng.integers(-2, L + 2, size=T).astype(np.int32)
        key = key_of(m, n, L)
        order = []
        for t in range(n):
            i = len(order)
            while i > 0 and key[order[i - 1]] > key[t]:
                i -= 1
            order.insert(i, t)
        s, c, st, status = oracle.prepare_metadata(m, n, L)
        assert s[:n].tolist() == order
        bad = np.any((m[:n] < -1) | (m[:n] >= L))
        assert status == (oracle.STATUS_BAD_LORA_ID if bad else 0)


def test_metadata_brute_force_all_tiny_mappings():
    # every mapping of 5 tokens over {-1, 0, 1}: the output must be the unique
    # permutation whose keys are non-decreasing with ties in token order
    L, T = 2, 5
    for mp in itertools.product([-1, 0, 1], repeat=T):
        m = np.array(mp, np.int32)
        s, c, st, status = oracle.prepare_metadata(m, T, L)
        key = key_of(m, T, L)
        found = None
        for p in itertools.permutations(range(T)):
            if all((key[p[i]], p[i]) < (key[p[i + 1]], p[i + 1]) for i in range(T - 1)):
                found = p
                break
        assert tuple(s.tolist()) == found
        assert status == 0
        for b in range(L + 1):
            assert c[b] == sum(1 for t in range(T) if key[t] == b)


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_metadata_invariants(name):
    shape = W.CONFIGS[name]
    m = W.make_mapping(shape, np.random.default_rng(1000 + shape.index))
    n, L = shape.num_tokens, shape.max_loras
    s, c, st, status = oracle.prepare_metadata(m, n, L)
    assert c.sum() == n and st[0] == 0 and st[-1] == n
    assert np.all(np.diff(st) >= 0)
    assert sorted(s[:n].tolist()) == list(range(n))
    for b in range(L + 1):
        seg = s[st[b]:st[b + 1]]
        assert np.all(np.diff(seg) > 0)
        if b < L:
            assert np.all(m[seg] == b)
    assert status == 0


def test_metadata_pad_entries_never_read_and_n_clamped():
    m = np.array([0, 1, 99, -7], np.int32)   # pad entries are out of range on purpose
    s, c, st, status = oracle.prepare_metadata(m, 2, 2)
    assert s.tolist() == [0, 1, -1, -1] and status == 0
    s, c, st, status = oracle.prepare_metadata(m, 9, 2)
    assert status & oracle.STATUS_BAD_NUM_TOKENS and st[-1] == 4
    s, c, st, status = oracle.prepare_metadata(m, -3, 2)
    assert status == oracle.STATUS_BAD_NUM_TOKENS and s.tolist() == [-1] * 4


# ---------------------------------------------------------------- shrink / expand

def test_gemm_worked_example():
    g = json.load(open(GOLDEN))["gemm"]
    x = bits(g["x"])
    a = [bits(g["lora_a"])]
    b = [bits(g["lora_b"])]
    y = bits(g["y_in"])
    m = np.array(g["token_lora_mapping"], np.int32)
    u = oracle.shrink(x, a, g["scale"], m, g["num_tokens"], g["max_loras"])
    for t, row in enumerate(g["u_expected"]):
        if row[0] is None:
            assert np.all(np.isnan(u[0, t]))
        else:
            assert u[0, t].tolist() == row
    yo = oracle.expand(np.nan_to_num(u), b, y, m, g["num_tokens"], g["max_loras"])
    assert yo.tolist() == [[float(v) for v in r] for r in g["y_expected"]]


def _random_layer(rng, T, H, widths, L, R, std=0.5):
    x = bits(rng.standard_normal((T, H)))
    a = [bits(std * rng.standard_normal((L, R, H))) for _ in widths]
    b = [bits(std * rng.standard_normal((L, R, w))) for w in widths]
    y = bits(rng.standard_normal((T, sum(widths))))
    return x, a, b, y


def test_shrink_one_adapter_equals_dense_numpy_matmul():
    rng = np.random.default_rng(11)
    T, H, widths, L, R = 37, 96, (24, 40, 16), 3, 8   # R != H, S = 3: catches transposes
    x, a, _, _ = _random_layer(rng, T, H, widths, L, R)
    for lid in range(L):
        m = np.full(T, lid, np.int32)
        u = oracle.shrink(x, a, 0.75, m, T, L)
        for s in range(len(widths)):
            dense = 0.75 * (val(x) @ val(a[s][lid]).T)
            np.testing.assert_allclose(u[s], dense, rtol=1e-12, atol=1e-12)


def test_shrink_mixed_batch_rows_equal_their_adapters_dense_result():
    rng = np.random.default_rng(12)
    T, H, widths, L, R = 50, 64, (32, 32), 4, 16
    x, a, _, _ = _random_layer(rng, T, H, widths, L, R)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    u = oracle.shrink(x, a, 1.0, m, T, L)
    for t in range(T):
        for s in range(2):
            if m[t] < 0:
                assert np.all(np.isnan(u[s, t]))
            else:
                ref = val(a[s][m[t]]) @ val(x[t])
                np.testing.assert_allclose(u[s, t], ref, rtol=1e-12, atol=1e-12)


def test_shrink_one_hot_row_selects_a_column_of_A():
    rng = np.random.default_rng(13)
    T, H, L, R = 6, 32, 2, 8
    _, a, _, _ = _random_layer(rng, T, H, (8,), L, R)
    x = np.zeros((T, H), np.float32)
    hs = [0, 5, 31, 17, 2, 9]
    for t, h in enumerate(hs):
        x[t, h] = 1.0
    m = np.array([0, 1, 1, 0, -1, 1], np.int32)
    u = oracle.shrink(bits(x), a, 2.0, m, T, L)
    for t, h in enumerate(hs):
        if m[t] >= 0:
            assert np.array_equal(u[0, t], 2.0 * val(a[0][m[t]][:, h]))


def test_shrink_scale_is_linear_and_zero_scale_gives_zero():
    rng = np.random.default_rng(14)
    T, H, L, R = 20, 48, 3, 8
    x, a, _, _ = _random_layer(rng, T, H, (8,), L, R)
    m = rng.integers(0, L, size=T).astype(np.int32)
    u1 = oracle.shrink(x, a, 1.0, m, T, L)
    uq = oracle.shrink(x, a, 0.25, m, T, L)
    u0 = oracle.shrink(x, a, 0.0, m, T, L)
    assert np.array_equal(uq, 0.25 * u1)       # power-of-two scale is exact
    assert np.all(u0 == 0.0)


def test_shrink_per_adapter_scales_match_dense_rows_and_the_scalar_path():
    """Per-adapter factors: each row equals the dense numpy product scaled
    by scale * factor of its adapter; factors of 1 give the scalar result."""
    rng = np.random.default_rng(15)
    T, H, widths, L, R = 40, 72, (16, 24), 4, 8
    x, a, _, _ = _random_layer(rng, T, H, widths, L, R)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    f = np.array([0.5, -2.0, 0.0, 3.25])
    u = oracle.shrink(x, a, 0.75, m, T, L, lora_scales=f)
    for t in range(T):
        for s in range(len(widths)):
            if m[t] < 0:
                assert np.all(np.isnan(u[s, t]))
            else:
                ref = 0.75 * f[m[t]] * (val(a[s][m[t]]) @ val(x[t]))
                np.testing.assert_allclose(u[s, t], ref, rtol=1e-12, atol=1e-12)
    ones = oracle.shrink(x, a, 0.75, m, T, L, lora_scales=np.ones(L))
    assert np.array_equal(ones, oracle.shrink(x, a, 0.75, m, T, L), equal_nan=True)


def test_shrink_leaves_unmapped_and_pad_rows_untouched():
    rng = np.random.default_rng(15)
    T, n, H, L, R = 16, 11, 32, 2, 8
    x, a, _, _ = _random_layer(rng, T, H, (8,), L, R)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    m[n:] = 0                                  # valid ids in the pad region
    init = np.full((1, T, R), 123.0)
    u = oracle.shrink(x, a, 1.0, m, n, L, u_init=init)
    for t in range(T):
        if t >= n or m[t] < 0:
            assert np.all(u[0, t] == 123.0)
        else:
            assert not np.any(u[0, t] == 123.0)


def test_expand_one_adapter_equals_dense_numpy_matmul():
    rng = np.random.default_rng(21)
    T, widths, L, R = 29, (40, 24, 56), 3, 16
    _, _, b, y = _random_layer(rng, T, 8, widths, L, R)
    u = rng.standard_normal((3, T, R))
    for lid in range(L):
        m = np.full(T, lid, np.int32)
        out = oracle.expand(u, b, y, m, T, L)
        dense = val(y) + np.concatenate([u[s] @ val(b[s][lid]) for s in range(3)], axis=1)
        np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12)


def test_expand_zero_B_keeps_y_and_zero_base_gives_the_delta():
    rng = np.random.default_rng(22)
    T, widths, L, R = 12, (16, 16), 2, 8
    _, _, b, y = _random_layer(rng, T, 8, widths, L, R)
    u = rng.standard_normal((2, T, R))
    m = rng.integers(-1, L, size=T).astype(np.int32)
    zb = [np.zeros_like(bb) for bb in b]
    assert np.array_equal(oracle.expand(u, zb, y, m, T, L), val(y))
    delta = oracle.expand(u, b, np.zeros_like(y), m, T, L)
    full = oracle.expand(u, b, y, m, T, L)
    np.testing.assert_allclose(full, val(y) + delta, rtol=1e-13, atol=1e-13)
    for t in range(T):
        if m[t] < 0:
            assert np.all(delta[t] == 0.0)


def test_expand_pad_rows_and_unmapped_rows_copy_y_exactly():
    rng = np.random.default_rng(23)
    T, n, widths, L, R = 10, 6, (16,), 2, 8
    _, _, b, y = _random_layer(rng, T, 8, widths, L, R)
    y_wide = np.concatenate([y, bits(np.full((T, 8), 3.0))], axis=1)   # row stride > sum N_s
    u = rng.standard_normal((1, T, R))
    m = np.array([0, -1, 1, 1, -1, 0, 0, 1, 1, 0], np.int32)
    out = oracle.expand(u, b, y_wide, m, n, L)
    for t in range(T):
        if t >= n or m[t] < 0:
            assert np.array_equal(out[t], val(y_wide[t]))
        else:
            assert np.array_equal(out[t, 16:], val(y_wide[t, 16:]))


def test_shrink_then_expand_is_associative():
    # y + (scale x A^T) B  ==  y + scale x (A^T B): the right side is computed
    # by numpy in the other association order
    rng = np.random.default_rng(31)
    T, H, widths, L, R = 40, 72, (24, 32), 3, 8
    x, a, b, y = _random_layer(rng, T, H, widths, L, R)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    u = oracle.shrink(x, a, 0.5, m, T, L)
    out = oracle.expand(np.nan_to_num(u), b, y, m, T, L)
    for t in range(T):
        if m[t] < 0:
            assert np.array_equal(out[t], val(y[t]))
            continue
        ab = np.concatenate([val(a[s][m[t]]).T @ val(b[s][m[t]]) for s in range(2)], axis=1)
        ref = val(y[t]) + 0.5 * (val(x[t]) @ ab)
        np.testing.assert_allclose(out[t], ref, rtol=1e-10, atol=1e-10)


def test_token_permutation_permutes_outputs_exactly():
    rng = np.random.default_rng(32)
    T, H, widths, L, R = 33, 40, (16,), 3, 8
    x, a, b, y = _random_layer(rng, T, H, widths, L, R)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    perm = rng.permutation(T)
    u = oracle.shrink(x, a, 1.0, m, T, L)
    up = oracle.shrink(x[perm], a, 1.0, m[perm], T, L)
    assert np.array_equal(np.nan_to_num(u[:, perm], nan=7.0), np.nan_to_num(up, nan=7.0))
    o = oracle.expand(np.nan_to_num(u), b, y, m, T, L)
    op = oracle.expand(np.nan_to_num(up), b, y[perm], m[perm], T, L)
    assert np.array_equal(o[perm], op)


def test_exact_small_integer_case_matches_integer_arithmetic():
    # every value and partial sum is a small integer (exact in bf16 and fp64),
    # so the oracle must equal int64 arithmetic exactly
    rng = np.random.default_rng(41)
    T, H, widths, L, R = 24, 16, (16, 8), 3, 8
    xi = rng.choice([-2, 0, 2], size=(T, H))
    ai = [rng.choice([-1, 0, 1], size=(L, R, H)) for _ in widths]
    bi = [rng.choice([-1, 0, 1], size=(L, R, w)) for w in widths]
    yi = rng.integers(-8, 9, size=(T, sum(widths)))
    m = rng.integers(-1, L, size=T).astype(np.int32)
    u = oracle.shrink(bits(xi), [bits(v) for v in ai], 0.5, m, T, L)
    out = oracle.expand(np.nan_to_num(u), [bits(v) for v in bi], bits(yi), m, T, L)
    for t in range(T):
        if m[t] < 0:
            assert np.array_equal(out[t], yi[t])
            continue
        uu = [ai[s][m[t]] @ xi[t] for s in range(2)]          # int64, scale applied below
        for s in range(2):
            assert np.array_equal(u[s, t] * 2, uu[s])
        delta = np.concatenate([uu[s] @ bi[s][m[t]] for s in range(2)])
        assert np.array_equal(out[t] * 2, 2 * yi[t] + delta)


def test_oracle_builds_with_threads():
    assert oracle.max_threads() >= 1


# ---------------------------------------------------------------- fp16 inputs

def test_decoders_match_numpy_on_every_bit_pattern():
    """Both 16-bit decoders against independent float conversions over all
    65536 patterns: fp16 against numpy's float16, bf16 against the top half
    of a float32 word; NaN patterns must decode to NaN."""
    every = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):   # widening signalling NaNs
        refs = ((True, every.view(np.float16).astype(np.float64)),
                (False, (every.astype(np.uint32) << 16).view(np.float32).astype(np.float64)))
    for f16, ref in refs:
        got = oracle.decode_bits(every, f16=f16)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])
    # a few fp16 values written out by hand: smallest subnormal, largest
    # subnormal, smallest normal, one, largest finite, negative two
    hand = {0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24, 0x0400: 2.0 ** -14,
            0x3C00: 1.0, 0x7BFF: 65504.0, 0xC000: -2.0}
    got = oracle.decode_bits(np.array(list(hand), np.uint16), f16=True)
    assert got.tolist() == list(hand.values())


def _f16_bits(a):
    return np.asarray(a, np.float16).view(np.uint16)


def test_fp16_shrink_and_expand_equal_dense_numpy_matmuls():
    """fp16 inputs: one-adapter rows of a mixed batch equal numpy's dense
    products on the same float16 values (a transposed operand or a bf16
    decoding of fp16 words fails this)."""
    rng = np.random.default_rng(21)
    T, H, widths, L, R = 30, 80, (24, 40), 3, 8
    x16 = rng.standard_normal((T, H)).astype(np.float16)
    a16 = [(0.5 * rng.standard_normal((L, R, H))).astype(np.float16) for _ in widths]
    b16 = [(0.5 * rng.standard_normal((L, R, w))).astype(np.float16) for w in widths]
    y16 = rng.standard_normal((T, sum(widths))).astype(np.float16)
    m = rng.integers(-1, L, size=T).astype(np.int32)
    u = oracle.shrink(_f16_bits(x16), [_f16_bits(v) for v in a16], 0.5, m, T, L, f16=True)
    y = oracle.expand(np.nan_to_num(u), [_f16_bits(v) for v in b16], _f16_bits(y16), m, T, L,
                      f16=True)
    x64, y64 = x16.astype(np.float64), y16.astype(np.float64)
    for t in range(T):
        off = 0
        for s, w in enumerate(widths):
            if m[t] < 0:
                assert np.all(np.isnan(u[s, t]))
                assert np.array_equal(y[t, off:off + w], y64[t, off:off + w])
            else:
                us = 0.5 * (a16[s][m[t]].astype(np.float64) @ x64[t])
                np.testing.assert_allclose(u[s, t], us, rtol=1e-12, atol=1e-12)
                ys = y64[t, off:off + w] + us @ b16[s][m[t]].astype(np.float64)
                np.testing.assert_allclose(y[t, off:off + w], ys, rtol=1e-12, atol=1e-12)
            off += w
