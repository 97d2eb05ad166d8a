"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- numbers printed on the pages, closed forms, invariants, an
independent numpy formulation, or a library routine on the cases where the
two must agree.  No GPU is used here."""
import math

import numpy as np
import pytest
import torch

import oracle

BS = oracle.BLOCK_SIZE


# ----------------------------------------------------------------- helpers

def bits_of(x):
    """float64/float32 values that are exactly bfloat16 -> uint16 patterns
    (via torch, the library conversion)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def build_paged(K, V, rng, num_blocks=None, kv_heads=1, head=0):
    """Place contiguous K, V [L, D] (bfloat16-exact values) into a paged pool
    [NB, Hkv, 16, D] under a random block permutation.  Unused slots get
    random finite values.  Returns (k_cache, v_cache, block_table_row)."""
    L, D = K.shape
    nb = -(-L // BS)
    NB = num_blocks or nb + 3
    perm = rng.permutation(NB)[:nb].astype(np.int32)
    kc = bits_of(rng.standard_normal((NB, kv_heads, BS, D)))
    vc = bits_of(rng.standard_normal((NB, kv_heads, BS, D)))
    kb, vb = bits_of(K), bits_of(V)
    for j in range(L):
        kc[perm[j // BS], head, j % BS] = kb[j]
        vc[perm[j // BS], head, j % BS] = vb[j]
    return kc, vc, perm


def bf16_exact(a):
    """Round an array to bfloat16 values (float64 out) with torch."""
    t = torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def run_oracle_single(q, kc, vc, bt_row, L, scale, kv_heads=1, G=1):
    B = 1
    qq = np.asarray(q, dtype=np.float64).reshape(B, kv_heads * G, -1)
    bt = np.asarray(bt_row, dtype=np.int32).reshape(1, -1)
    cl = np.array([L], dtype=np.int32)
    return oracle.paged_attention(qq, kc, vc, bt, cl, scale)


# --------------------------------------------------------------- kv_bytes

def test_kv_bytes_worked_examples(golden):
    rows = golden("kv_bytes_examples.txt")
    assert len(rows) == 6
    for layers, batch, heads, seq, d, nbytes, expected in rows:
        assert oracle.kv_bytes(layers, batch, heads, seq, d, nbytes) == expected


def test_kv_bytes_linear_in_each_factor():
    base = oracle.kv_bytes(32, 32, 8, 8192, 128, 2)
    # "doubling the sequence doubles the cache" (mask/KV-cache page, memory section)
    assert oracle.kv_bytes(32, 32, 8, 16384, 128, 2) == 2 * base
    # GQA 32 -> 8 KV heads is a 4x reduction ("(2) GQA" section)
    assert oracle.kv_bytes(32, 32, 32, 8192, 128, 2) == 4 * base
    # FP8 halves it ("(1) FP8 quantization" section)
    assert 2 * oracle.kv_bytes(32, 32, 8, 8192, 128, 1) == base


# ----------------------------------------------------------- slot mapping

def test_slot_mapping_hand_example(golden):
    rows = golden("slot_mapping_example.txt")
    bt = np.array([[7, 2, 9]], dtype=np.int32)
    pos = np.array([r[0] for r in rows])
    want = np.array([r[1] for r in rows])
    got = oracle.slot_mapping(bt, np.zeros_like(pos), pos)
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------------- attention

def test_single_key_returns_that_value():
    rng = np.random.default_rng(1)
    D = 64
    K = bf16_exact(rng.standard_normal((1, D)))
    V = bf16_exact(rng.standard_normal((1, D)))
    kc, vc, bt = build_paged(K, V, rng)
    q = bf16_exact(rng.standard_normal(D))
    out = run_oracle_single(q, kc, vc, bt, 1, 0.125)
    np.testing.assert_array_equal(out[0, 0], V[0])


def test_rows_are_probability_vectors():
    # with V_j = e_j the output is the softmax weight vector itself
    rng = np.random.default_rng(2)
    L, D = 50, 64
    K = bf16_exact(rng.standard_normal((L, D)))
    V = np.eye(L, D)
    kc, vc, bt = build_paged(K, V, rng)
    q = bf16_exact(rng.standard_normal(D))
    w = run_oracle_single(q, kc, vc, bt, L, 0.125)[0, 0, :L]
    assert np.all(w > 0)
    assert abs(w.sum() - 1.0) < 1e-12
    # and the weights are the softmax of the scores (closed form)
    z = 0.125 * (K @ q)
    np.testing.assert_allclose(w, np.exp(z - z.max()) / np.exp(z - z.max()).sum(), rtol=1e-12)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    L, D = 37, 128
    k = bf16_exact(rng.standard_normal(D))
    K = np.tile(k, (L, 1))
    V = bf16_exact(rng.standard_normal((L, D)))
    kc, vc, bt = build_paged(K, V, rng)
    q = bf16_exact(rng.standard_normal(D))
    out = run_oracle_single(q, kc, vc, bt, L, 1 / math.sqrt(D))
    np.testing.assert_allclose(out[0, 0], V.mean(axis=0), rtol=0, atol=1e-12)


def test_zero_keys_give_uniform_average():
    rng = np.random.default_rng(4)
    L, D = 23, 64
    K = np.zeros((L, D))
    V = bf16_exact(rng.standard_normal((L, D)))
    kc, vc, bt = build_paged(K, V, rng)
    q = bf16_exact(rng.standard_normal(D))
    out = run_oracle_single(q, kc, vc, bt, L, 0.125)
    np.testing.assert_allclose(out[0, 0], V.mean(axis=0), rtol=0, atol=1e-12)


def test_dominant_score_selects_its_value():
    rng = np.random.default_rng(5)
    L, D, t = 40, 64, 29
    K = bf16_exact(rng.standard_normal((L, D)))
    q = np.zeros(D)
    q[3] = 64.0
    K[t] = 0.0
    K[t, 3] = 64.0                       # score 64*64/8 = 512, others ~ 8
    V = bf16_exact(rng.standard_normal((L, D)))
    kc, vc, bt = build_paged(K, V, rng)
    out = run_oracle_single(q, kc, vc, bt, L, 0.125)
    np.testing.assert_allclose(out[0, 0], V[t], rtol=0, atol=1e-12)


def test_output_is_convex_combination():
    rng = np.random.default_rng(6)
    L, D = 300, 128
    K = bf16_exact(rng.standard_normal((L, D)))
    V = bf16_exact(rng.standard_normal((L, D)))
    kc, vc, bt = build_paged(K, V, rng)
    q = bf16_exact(rng.standard_normal(D))
    out = run_oracle_single(q, kc, vc, bt, L, 1 / math.sqrt(D))[0, 0]
    assert np.all(out <= V.max(axis=0) + 1e-12)
    assert np.all(out >= V.min(axis=0) - 1e-12)


def test_paged_equals_contiguous_and_permutation_invariant():
    rng = np.random.default_rng(7)
    L, D = 97, 128
    K = bf16_exact(rng.standard_normal((L, D)))
    V = bf16_exact(rng.standard_normal((L, D)))
    q = bf16_exact(rng.standard_normal(D))
    ref = oracle.attention_direct(q, K, V, 1 / math.sqrt(D))
    outs = []
    for trial in range(3):
        kc, vc, bt = build_paged(K, V, np.random.default_rng(100 + trial), num_blocks=20)
        outs.append(run_oracle_single(q, kc, vc, bt, L, 1 / math.sqrt(D))[0, 0])
    np.testing.assert_allclose(outs[0], ref, rtol=0, atol=1e-13)
    # the gather makes the arithmetic order independent of the physical layout
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


@pytest.mark.parametrize("L", [1, 2, 5, 16, 17, 33, 64])
def test_decode_equals_last_row_of_causal_attention(L):
    rng = np.random.default_rng(10 + L)
    D = 64
    Q = bf16_exact(rng.standard_normal((L, D)))
    K = bf16_exact(rng.standard_normal((L, D)))
    V = bf16_exact(rng.standard_normal((L, D)))
    full = oracle.causal_attention(Q, K, V, 0.125)
    kc, vc, bt = build_paged(K, V, rng)
    dec = run_oracle_single(Q[L - 1], kc, vc, bt, L, 0.125)[0, 0]
    np.testing.assert_allclose(dec, full[L - 1], rtol=0, atol=1e-12)
    # every earlier row is itself a decode step over its own prefix
    t = L // 2
    dec_t = run_oracle_single(Q[t], kc, vc, bt, t + 1, 0.125)[0, 0]
    np.testing.assert_allclose(dec_t, full[t], rtol=0, atol=1e-12)


def test_causal_mask_matches_page(golden):
    want = np.array(golden("causal_mask_4.txt"), dtype=bool)
    got = oracle.causal_mask(4) == 0.0
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("L", [1, 3, 4, 7, 64, 129])
def test_tiled_running_softmax_equals_direct(L):
    rng = np.random.default_rng(200 + L)
    D = 32
    q = rng.standard_normal(D)
    K = rng.standard_normal((L, D)) * 3.0
    V = rng.standard_normal((L, D))
    direct = oracle.attention_direct(q, K, V, 0.5)
    for tile in (1, 4, 16):
        tiled = oracle.tiled_softmax_attention(q, K, V, 0.5, tile=tile)
        np.testing.assert_allclose(tiled, direct, rtol=0, atol=1e-12)


def test_padding_keys_have_no_influence():
    # a real length of 3 inside a padded block of 5+ ([A, B, C, PAD, PAD]):
    # whatever sits in the PAD slots must not change the result
    rng = np.random.default_rng(11)
    D = 64
    K = bf16_exact(rng.standard_normal((3, D)))
    V = bf16_exact(rng.standard_normal((3, D)))
    q = bf16_exact(rng.standard_normal(D))
    kc, vc, bt = build_paged(K, V, rng)
    base = run_oracle_single(q, kc, vc, bt, 3, 0.125)[0, 0]
    nan_bits = np.uint16(0x7FC0)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[bt[0], 0, 3:] = nan_bits
    vc2[bt[0], 0, 3:] = nan_bits
    pad = run_oracle_single(q, kc2, vc2, bt, 3, 0.125)[0, 0]
    np.testing.assert_array_equal(base, pad)
    np.testing.assert_allclose(base, oracle.attention_direct(q, K, V, 0.125), atol=1e-13)


def test_gqa_group_reads_its_kv_head():
    # query head h uses KV head h // G: permuting KV heads permutes the
    # query-head groups of the output
    rng = np.random.default_rng(12)
    Hkv, G, D, L = 3, 2, 64, 40
    NB = 4
    kc = bits_of(rng.standard_normal((NB, Hkv, BS, D)))
    vc = bits_of(rng.standard_normal((NB, Hkv, BS, D)))
    q = bf16_exact(rng.standard_normal((1, Hkv * G, D)))
    bt = np.array([[2, 0, 3]], dtype=np.int32)
    cl = np.array([L], dtype=np.int32)
    out = oracle.paged_attention(q, kc, vc, bt, cl, 0.125)
    for h in range(Hkv * G):
        hk = h // G
        Kc = np.concatenate([oracle.bf16_bits_to_f64(kc[b, hk]) for b in bt[0]])[:L]
        Vc = np.concatenate([oracle.bf16_bits_to_f64(vc[b, hk]) for b in bt[0]])[:L]
        np.testing.assert_allclose(out[0, h], oracle.attention_direct(q[0, h], Kc, Vc, 0.125),
                                   atol=1e-13)


def test_empty_context_defined_as_zero():
    rng = np.random.default_rng(13)
    kc = bits_of(rng.standard_normal((2, 1, BS, 64)))
    out = oracle.paged_attention(np.ones((1, 2, 64)), kc, kc.copy(),
                                 np.array([[-1]], dtype=np.int32),
                                 np.array([0], dtype=np.int32), 0.125)
    assert np.all(out == 0.0)


def test_pair_select_computes_only_selected_pairs():
    rng = np.random.default_rng(14)
    kc = bits_of(rng.standard_normal((4, 2, BS, 64)))
    vc = bits_of(rng.standard_normal((4, 2, BS, 64)))
    q = bf16_exact(rng.standard_normal((2, 4, 64)))
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    cl = np.array([20, 31], dtype=np.int32)
    full = oracle.paged_attention(q, kc, vc, bt, cl, 0.125)
    sel = np.array([[False, True], [True, False]])
    part = oracle.paged_attention(q, kc, vc, bt, cl, 0.125, pair_select=sel)
    np.testing.assert_array_equal(part[0, 2:], full[0, 2:])
    np.testing.assert_array_equal(part[1, :2], full[1, :2])
    assert np.isnan(part[0, :2]).all() and np.isnan(part[1, 2:]).all()


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_matches_library_on_float32_inputs():
    rng = np.random.default_rng(20)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),     # binary32 subnormals
        (rng.uniform(-1, 1, 2000) * 3e38).astype(np.float32),
        np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 2**-126 * (1 + 2**-8),
                  3.3895314e38, 3.4e38, 0.0, -0.0, np.inf, -np.inf], dtype=np.float32),
    ])
    want = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_ties_to_even_and_roundtrip():
    assert oracle.f64_to_bf16_bits(np.array([1 + 2**-8]))[0] == 0x3F80      # tie -> 1.0
    assert oracle.f64_to_bf16_bits(np.array([1 + 3 * 2**-8]))[0] == 0x3F82  # tie -> even
    assert oracle.f64_to_bf16_bits(np.array([1 + 2**-8 + 2**-30]))[0] == 0x3F81
    bits = np.arange(65536, dtype=np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    np.testing.assert_array_equal(oracle.f64_to_bf16_bits(vals[finite]), bits[finite])


# ------------------------------------------------------------------ E4M3

def test_e4m3_decode_closed_forms():
    d = oracle.e4m3_decode
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert d(0x38) == 1.0
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x08) == 2.0**-6              # smallest normal
    assert d(0x01) == 2.0**-9              # smallest subnormal
    assert d(0x07) == 7 * 2.0**-9          # largest subnormal
    assert d(0x77) == 240.0                # 1.875 * 2^7
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert not math.isinf(d(0x78))         # no infinities: 0x78 = 256
    assert d(0x78) == 256.0
    # exactly 254 finite codes, strictly increasing over the positive half
    pos = [d(c) for c in range(0x00, 0x7F)]
    assert all(b > a for a, b in zip(pos, pos[1:]))


def test_e4m3_encode_roundtrip_every_code():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_ties_and_saturation():
    e = oracle.e4m3_encode
    assert e(1.0 + 1 / 16) == 0x38          # halfway 1.0 / 1.125 -> even (1.0)
    assert e(1.0 + 3 / 16) == 0x3A          # halfway 1.125 / 1.25 -> even (1.25)
    assert e(1.0 + 1 / 16 + 1e-9) == 0x39
    assert e(2.0**-10) == 0x00              # half the smallest subnormal -> 0
    assert e(3 * 2.0**-10) == 0x02          # halfway 1 / 2 subnormal units -> 2
    assert e(-3 * 2.0**-10) == 0x82
    assert e(-1e-6) == 0x80                 # underflow keeps the sign
    assert e(464.0) == 0x7E                 # would round to 480: saturates
    assert e(1e9) == 0x7E and e(-1e9) == 0xFE
    assert e(float("inf")) == 0x7E and e(float("-inf")) == 0xFE
    assert e(float("nan")) & 0x7F == 0x7F
    assert e(7.5 * 2.0**-9) == 0x08         # halfway largest subnormal / min normal -> even
    assert e(0.0) == 0x00


def test_e4m3_encode_is_nearest():
    # against brute force: nearest finite code by distance, ties to even code
    finite = [(c, oracle.e4m3_decode(c)) for c in range(0x7F)]
    rng = np.random.default_rng(21)
    xs = np.concatenate([rng.uniform(0, 460, 3000), rng.uniform(0, 0.05, 3000)])
    for x in xs:
        best = min(finite, key=lambda cv: (abs(cv[1] - x), cv[0] & 1))
        if x > 448:
            best = (0x7E, 448.0)
        assert oracle.e4m3_encode(x) == best[0], x


def _e4m3_finite_values():
    """(value, code) of every non-negative finite E4M3 ("fn") number, from the
    format's definition: 4 exponent bits (bias 7), 3 mantissa bits,
    subnormals at exponent field 0, S.1111.111 reserved for NaN."""
    from fractions import Fraction
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            if e == 0:
                v = Fraction(m, 8) * Fraction(1, 2 ** 6)
            else:
                v = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
            vals.append((v, (e << 3) | m))
    return sorted(vals)


def _exact_e4m3_codes(x, scale):
    """E4M3 code of the exact real quotient x / scale for every float in x:
    nearest finite value, ties to the even code, saturation to +-448.  x is
    compared with the midpoints scaled by `scale` (x / s > mid <=> x > mid * s
    for s > 0), all in exact rational arithmetic."""
    import bisect
    from fractions import Fraction
    vals = _e4m3_finite_values()
    s = Fraction(float(scale))
    thr = [(vals[i][0] + vals[i + 1][0]) / 2 * s for i in range(len(vals) - 1)]
    top = vals[-1][0] * s                       # 448 * s: saturation from here up
    codes = np.empty(len(x), dtype=np.uint8)
    for n, xv in enumerate(x):
        a = Fraction(abs(float(xv)))
        if a >= top:
            c = vals[-1][1]
        else:
            i = bisect.bisect_left(thr, a)      # thr[i-1] < a <= thr[i]
            if i < len(thr) and a == thr[i]:    # exactly halfway: the even code
                lo, hi = vals[i][1], vals[i + 1][1]
                c = lo if lo % 2 == 0 else hi
            else:
                c = vals[i][1]
        codes[n] = c | (0x80 if math.copysign(1.0, float(xv)) < 0 else 0)
    return codes


# 4.75/448 and 7.0 are scales at which multiplying by a binary32 reciprocal
# instead of dividing changes some codes; 1/3 and 0.1 have binary32 quotients
# that land on E4M3 midpoints
@pytest.mark.parametrize("scale", [1.0, 4.25 / 448, 4.75 / 448, 1.0 / 3, 0.1, 3.0 * 2.0**-20,
                                   7.0])
def test_quantize_agrees_with_exact_real_quotient(scale):
    """The stored code of x is E4M3(x / scale), x a bfloat16 value and scale
    a binary32 number ("KV cache complete guide", section "(1) FP8
    quantization": a per-tensor scale; the plainest encoding).  Here the
    quotient is the exact real number (Python fractions) and E4M3 is taken
    from its definition, over every finite bfloat16.  The oracle forms the
    quotient in binary32 first, as the writing kernel does.  Because every
    E4M3 value and midpoint is a binary32 number and rounding is monotone,
    that changes the result exactly where the binary32 quotient lands on a
    midpoint that the exact quotient misses, on the side of an odd code:
    the oracle then takes the even neighbour.  The test computes that set
    on its own and asserts that the oracle differs from the exact code on
    that set and nowhere else."""
    from fractions import Fraction
    scale = float(np.float32(scale))
    bits = np.arange(65536, dtype=np.uint16)
    x = oracle.bf16_bits_to_f64(bits)
    fin = np.isfinite(x)
    bits, x = bits[fin], x[fin]
    got = oracle.quantize_e4m3(bits, scale)
    want = _exact_e4m3_codes(x, scale)
    vals = _e4m3_finite_values()
    mids = {float((a[0] + b[0]) / 2): (a[1], b[1]) for a, b in zip(vals[:-1], vals[1:])}
    with np.errstate(over="ignore"):
        q32 = np.abs(x.astype(np.float32) / np.float32(scale)).astype(np.float64)
    expect = set()
    for n in np.nonzero(np.isin(q32, list(mids)))[0]:
        lo, hi = mids[float(q32[n])]
        qx = Fraction(abs(float(x[n]))) / Fraction(scale)
        qf = Fraction(float(q32[n]))
        side = hi if qx > qf else lo if qx < qf else None
        if side is not None and side % 2 == 1:
            expect.add(int(n))
    differ = set(np.nonzero(got != want)[0].tolist())
    assert differ == expect, sorted(differ ^ expect)[:10]
    for n in differ:
        assert int(got[n]) % 2 == 0 and abs(int(got[n]) - int(want[n])) == 1
    print("scale %r: %d of %d finite bfloat16 values round twice through the binary32 "
          "quotient: %s" % (scale, len(differ), len(x),
                            [(hex(int(bits[n])), float(x[n])) for n in sorted(differ)[:6]]))
    if scale == 1.0:
        assert not differ                     # the quotient is exact


# ---------------------------------------------------------------- append

@pytest.mark.parametrize("kv_dtype", [oracle.BF16, oracle.FP8_E4M3])
def test_append_writes_exactly_the_slots(kv_dtype):
    rng = np.random.default_rng(30)
    NB, Hkv, D, T = 6, 2, 64, 5
    dt = np.uint16 if kv_dtype == oracle.BF16 else np.uint8
    canary = dt(0x5A5A if dt is np.uint16 else 0x5A)
    kc = np.full((NB, Hkv, BS, D), canary, dtype=dt)
    vc = kc.copy()
    k = bits_of(rng.standard_normal((T, Hkv, D)))
    v = bits_of(rng.standard_normal((T, Hkv, D)))
    slots = np.array([17, -1, 95, 0, 40], dtype=np.int64)
    ks, vs = 0.01, 0.02
    assert oracle.append(kc, vc, k, v, slots, kv_dtype, ks, vs) == 0
    touched = np.zeros((NB, BS), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), BS)
        touched[b, o] = True
        if kv_dtype == oracle.BF16:
            np.testing.assert_array_equal(kc[b, :, o], k[t])
            np.testing.assert_array_equal(vc[b, :, o], v[t])
        else:
            np.testing.assert_array_equal(kc[b, :, o], oracle.quantize_e4m3(k[t], ks))
            np.testing.assert_array_equal(vc[b, :, o], oracle.quantize_e4m3(v[t], vs))
    untouched = ~touched[:, None, :]          # broadcast over KV heads
    assert np.all(kc[np.broadcast_to(untouched, (NB, Hkv, BS))] == canary)
    assert np.all(vc[np.broadcast_to(untouched, (NB, Hkv, BS))] == canary)


def test_append_rejects_slot_outside_pool():
    kc = np.zeros((2, 1, BS, 8), dtype=np.uint16)
    vc = kc.copy()
    k = np.zeros((1, 1, 8), dtype=np.uint16)
    assert oracle.append(kc, vc, k, k, np.array([32]), oracle.BF16) == -1


def test_fp8_attention_reads_dequantised_values():
    rng = np.random.default_rng(31)
    L, D = 45, 64
    Kf = rng.standard_normal((L, D))
    Vf = rng.standard_normal((L, D))
    ks, vs = 4.0 / 448, 3.0 / 448
    kq = oracle.quantize_e4m3(bits_of(Kf), ks)
    vq = oracle.quantize_e4m3(bits_of(Vf), vs)
    NB = 5
    perm = rng.permutation(NB)[:3].astype(np.int32)
    kc = np.zeros((NB, 1, BS, D), dtype=np.uint8)
    vc = np.zeros((NB, 1, BS, D), dtype=np.uint8)
    for j in range(L):
        kc[perm[j // BS], 0, j % BS] = kq[j]
        vc[perm[j // BS], 0, j % BS] = vq[j]
    q = bf16_exact(rng.standard_normal(D))
    out = oracle.paged_attention(q.reshape(1, 1, D), kc, vc, perm.reshape(1, -1),
                                 np.array([L], dtype=np.int32), 0.125,
                                 kv_dtype=oracle.FP8_E4M3, k_scale=ks, v_scale=vs)[0, 0]
    Kd = oracle.e4m3_decode_array(kq) * ks
    Vd = oracle.e4m3_decode_array(vq) * vs
    np.testing.assert_allclose(out, oracle.attention_direct(q, Kd, Vd, 0.125), atol=1e-13)
    # and quantisation error against the unquantised values is small
    ref = oracle.attention_direct(q, bf16_exact(Kf), bf16_exact(Vf), 0.125)
    assert np.max(np.abs(out - ref)) < 0.1


# ------------------------------------------------- cached vs naive decoding

def test_token_by_token_generation_cached_equals_naive(golden):
    """A 100-token generation run both ways: the naive decoder recomputes
    causal attention over the whole prefix at every step, the cached one
    appends the new K/V into a paged pool (slots from the block table) and
    attends only the new query.  The pages fix the work of each (query rows
    attended) and require the two paths to give the same outputs."""
    (N, naive_want, cached_want), = golden("attention_op_count.txt")
    rng = np.random.default_rng(77)
    D, scale = 16, 0.25
    Q = bf16_exact(rng.standard_normal((N, D)))
    K = bf16_exact(rng.standard_normal((N, D)))
    V = bf16_exact(rng.standard_normal((N, D)))
    nb = -(-N // BS)
    NB = nb + 5
    bt = rng.permutation(NB)[:nb].astype(np.int32).reshape(1, nb)
    kc = bits_of(rng.standard_normal((NB, 1, BS, D)))     # stale contents everywhere
    vc = bits_of(rng.standard_normal((NB, 1, BS, D)))
    naive_ops = cached_ops = 0
    for t in range(N):
        rows = oracle.causal_attention(Q[:t + 1], K[:t + 1], V[:t + 1], scale)
        naive_ops += rows.shape[0]
        slot = oracle.slot_mapping(bt, [0], [t])
        assert oracle.append(kc, vc, bits_of(K[t]).reshape(1, 1, D),
                             bits_of(V[t]).reshape(1, 1, D), slot, oracle.BF16) == 0
        out = run_oracle_single(Q[t], kc, vc, bt[0], t + 1, scale)
        cached_ops += 1
        np.testing.assert_allclose(out[0, 0], rows[t], rtol=0, atol=1e-12)
    assert (naive_ops, cached_ops) == (naive_want, cached_want)
    assert naive_ops == N * (N + 1) // 2


# ---------------------------------------------------- split-KV and the merge

@pytest.mark.parametrize("L", [1, 17, 100, 513])
def test_split_partials_merge_to_direct_attention(L):
    """Any cut of the keys, empty ranges included, merged by log-sum-exp,
    equals one-shot attention; one range is the library's logsumexp."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(300 + L)
    D = 32
    q = rng.standard_normal(D)
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    scale = 0.3
    direct = oracle.attention_direct(q, K, V, scale)
    (o1, lse1), = oracle.split_partials(q, K, V, scale, [0, L])
    np.testing.assert_allclose(o1, direct, rtol=0, atol=1e-13)
    assert abs(lse1 - logsumexp(scale * (K @ q))) < 1e-12
    for trial in range(5):
        cuts = np.sort(rng.integers(0, L + 1, size=rng.integers(1, 9)))
        bounds = [0] + [int(c) for c in cuts] + [L]      # repeats give empty ranges
        parts = oracle.split_partials(q, K, V, scale, bounds)
        merged = oracle.lse_merge(parts)
        np.testing.assert_allclose(merged, direct, rtol=0, atol=1e-12)
        perm = rng.permutation(len(parts))
        np.testing.assert_allclose(oracle.lse_merge([parts[i] for i in perm]), merged,
                                   rtol=0, atol=1e-14)


def test_merge_is_stable_for_large_scores_and_empty_inputs():
    """Scores near 1e3 overflow e^z; the merge must still equal the direct
    result.  With no keys at all the merge gives zeros (the empty-context
    reading)."""
    rng = np.random.default_rng(310)
    D, L = 16, 64
    q = rng.standard_normal(D) * 40
    K = rng.standard_normal((L, D)) * 40
    V = rng.standard_normal((L, D))
    direct = oracle.attention_direct(q, K, V, 1.0)
    assert np.all(np.isfinite(direct))
    merged = oracle.lse_merge(oracle.split_partials(q, K, V, 1.0, [0, 10, 30, 31, 64]))
    np.testing.assert_allclose(merged, direct, rtol=0, atol=1e-12)
    empty = oracle.split_partials(q, K[:0], V[:0], 1.0, [0, 0, 0])
    np.testing.assert_array_equal(oracle.lse_merge(empty), np.zeros(D))
