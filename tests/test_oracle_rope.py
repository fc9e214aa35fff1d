"""Pins of the oracle's rotary embedding and fused paged append (CPU only).

What pins them, other than the formula itself:
  * closed forms: with D = 2 the embedding is a plain rotation of (x0, x1) by
    the position; with D = 4 and base 10000 the second pair turns at 1/100 of
    that rate; position 0 is the identity;
  * invariants of a rotation: each (x_i, x_{i+D/2}) pair keeps its length,
    dot products of a query and a key depend only on the position difference,
    and two rotations compose into one;
  * the bf16 rounding against torch's float32 -> bfloat16 conversion, and
    against bit patterns worked out by hand for f64 inputs that rounding
    through f32 first would get wrong (1 + 2^-8 + 2^-30 lies above the
    halfway point between two bf16 neighbours, but its f32 rounding lands
    exactly on it), for ties, for subnormal results (steps of 2^-133) and
    for overflow to infinity;
  * the append against a dense logical view of the cache built here with plain
    indexing (no page arithmetic from the oracle), and the write rule (pages
    whose reference count is not one stay untouched);
  * planted mistakes (split-half vs interleaved pairing, sign, frequency
    exponent, slot arithmetic, the reference-count rule, bf16 rounding through
    f32, truncated or missing subnormal rounding) are each rejected by this
    battery.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oxd_oracle.c")


def _bits(x):
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ the pin battery

# f64 value -> bf16 pattern, each worked out by hand. bf16 = sign | 8-bit
# exponent (bias 127) | 7-bit fraction; the smallest normal is 2^-126 (0x0080),
# subnormals are k * 2^-133 (pattern k), the largest finite value is
# (2 - 2^-7) * 2^127 (0x7F7F).
BF16_GOLDEN = [
    (1.0, 0x3F80),
    (1 + 2**-8 + 2**-30, 0x3F81),      # above the 1 | 1 + 2^-7 midpoint: up
    (-(1 + 2**-8 + 2**-30), 0xBF81),
    (1 + 2**-8, 0x3F80),               # the midpoint itself: to the even 1.0
    (1 + 3 * 2**-8, 0x3F82),           # midpoint of 1 + 2^-7, 1 + 2^-6: to even
    (1 + 3 * 2**-8 - 2**-40, 0x3F81),  # just below that midpoint: down
    (3.0 * 2**-127, 0x0040 | 0x0080),  # 1.5 * 2^-126 is normal: 0x00C0
    (2**-133, 0x0001),                 # the smallest subnormal
    (-(2**-133), 0x8001),
    (2**-134, 0x0000),                 # half of it: to the even 0
    (3 * 2**-134, 0x0002),             # 1.5 steps: to the even 2
    (2**-134 + 2**-150, 0x0001),       # just above half a step: up
    (127.5 * 2**-133, 0x0080),         # halfway to the smallest normal: to even (128)
    (126.5 * 2**-133, 0x007E),         # halfway between 126 and 127 steps: to even
    (5e-324, 0x0000),                  # the smallest f64 subnormal
    (255 * 2.0**120, 0x7F7F),          # the largest finite bf16
    ((2 - 2**-8) * 2.0**127, 0x7F80),  # midpoint of the largest and 2^128: to even (inf)
    ((2 - 2**-8) * 2.0**127 - 2.0**90, 0x7F7F),
    (1e300, 0x7F80),
    (-1e300, 0xFF80),
]


def bf16_pins(lib):
    """The hand-worked rounding cases; returns a list of failures."""
    bad = []
    for x, want in BF16_GOLDEN:
        got = int(oracle.f64_to_bf16(np.array([x]), lib=lib)[0])
        if got != want:
            bad.append(f"bf16({x!r}) = {got:#06x}, want {want:#06x}")
    return bad


def rope_pins(lib):
    """Every pin of the embedding; returns a list of failures (empty = pass)."""
    bad = []
    rng = np.random.default_rng(7)
    # position 0 is the identity
    x = rng.standard_normal((5, 128))
    if not np.array_equal(oracle.rope(x, np.zeros(5, np.int32), lib=lib), x):
        bad.append("position 0 is not the identity")
    # D = 2: a rotation of (x0, x1) by the position itself
    for p in (1, 3, 100, 32767):
        y = oracle.rope(np.array([[1.0, 0.0], [0.0, 1.0]]), [p, p], lib=lib)
        want = np.array([[math.cos(p), math.sin(p)], [-math.sin(p), math.cos(p)]])
        if not np.allclose(y, want, rtol=0, atol=1e-12):
            bad.append(f"D=2 is not a rotation by the position ({p})")
    # D = 4, base 10000: pairs (0, 2) at rate 1 and (1, 3) at rate 1/100
    for p in (7, 1234):
        y = oracle.rope(np.array([[0.0, 1.0, 0.0, 0.0]]), [p], lib=lib)[0]
        want = [0.0, math.cos(p / 100.0), 0.0, math.sin(p / 100.0)]
        if not np.allclose(y, want, rtol=0, atol=1e-12):
            bad.append(f"D=4 second frequency wrong ({p})")
    # lengths of the (i, i + D/2) pairs are preserved
    pos = rng.integers(0, 32768, 5).astype(np.int32)
    y = oracle.rope(x, pos, lib=lib)
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = y[:, :64] ** 2 + y[:, 64:] ** 2
    if not np.allclose(n0, n1, rtol=1e-12, atol=1e-12):
        bad.append("pair lengths not preserved")
    # q . k depends only on the position difference
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    for m, n, s in ((10, 3, 500), (0, 7, 20000), (300, 300, 1)):
        d0 = float((oracle.rope(q, [m], lib=lib) @ oracle.rope(k, [n], lib=lib).T)[0, 0])
        d1 = float((oracle.rope(q, [m + s], lib=lib) @ oracle.rope(k, [n + s], lib=lib).T)[0, 0])
        if not math.isclose(d0, d1, rel_tol=1e-9, abs_tol=1e-9):
            bad.append(f"dot product depends on absolute positions ({m}, {n}, {s})")
    # two rotations compose
    a, b = 123, 4567
    y2 = oracle.rope(oracle.rope(x[:1], [a], lib=lib), [b], lib=lib)
    if not np.allclose(y2, oracle.rope(x[:1], [a + b], lib=lib), rtol=1e-9, atol=1e-9):
        bad.append("rotations do not compose")
    return bad


def _tables():
    # two requests, page size 4: request 0 owns pages [5, 2, 7] (11 tokens,
    # growing to 12), request 1 owns pages [0, 3] (5 tokens, growing to 6);
    # page 3 is shared (reference count 2) in the second scenario
    indptr = np.array([0, 3, 5], np.int32)
    indices = np.array([5, 2, 7, 0, 3], np.int32)
    return indptr, indices


def append_pins(lib):
    """Every pin of the fused append; returns a list of failures."""
    bad = []
    rng = np.random.default_rng(11)
    ps, Hq, Hkv, D, num_pages = 4, 4, 2, 128, 9
    indptr, indices = _tables()
    for layout in (oracle.LAYOUT_NHD, oracle.LAYOUT_HND):
        shape = (num_pages, ps, Hkv, D) if layout == oracle.LAYOUT_NHD else (num_pages, Hkv, ps, D)
        k_pages = _bits(rng.standard_normal(shape))
        v_pages = _bits(rng.standard_normal(shape))
        T = 4
        q = _bits(rng.standard_normal((T, Hq, D)))
        k = _bits(rng.standard_normal((T, Hkv, D)))
        v = _bits(rng.standard_normal((T, Hkv, D)))
        # tokens: request 0 at position 11 (page 7, slot 3), request 1 at 5
        # (page 3, slot 1), request 1 at 4 (page 3, slot 0), request 0 at 12
        # (past its pages: not written)
        tr = np.array([0, 1, 1, 0], np.int32)
        pos = np.array([11, 5, 4, 12], np.int32)
        for shared in (False, True):
            rc = np.ones(num_pages, np.int32)
            if shared:
                rc[3] = 2
            q_out, kp, vp, st = oracle.rope_append(q, k, v, tr, pos, indptr, indices, rc,
                                                   k_pages, v_pages, page_size=ps, layout=layout,
                                                   lib=lib)
            want_st = [0, 1 if shared else 0, 1 if shared else 0, 2]
            if list(st) != want_st:
                bad.append(f"status {list(st)} != {want_st} (layout {layout}, shared {shared})")
            # q_out of every token, written or not
            want_q = oracle.f64_to_bf16(
                oracle.rope(_f64(q).reshape(-1, D), np.repeat(pos, Hq), lib=lib).reshape(q.shape))
            if not np.array_equal(q_out, want_q):
                bad.append("q_out is not bf16(RoPE(q))")
            # dense logical views of both pools, before and after
            def view(pool, page, slot, h):
                if layout == oracle.LAYOUT_NHD:
                    return pool[page, slot, h]
                return pool[page, h, slot]
            changed = set()
            for t in range(T):
                if want_st[t] != 0:
                    continue
                b, p = int(tr[t]), int(pos[t])
                page = int(indices[indptr[b] + p // ps])
                for h in range(Hkv):
                    changed.add((page, p % ps, h))
                    want_k = oracle.f64_to_bf16(oracle.rope(_f64(k[t, h])[None], [p], lib=lib)[0])
                    if not np.array_equal(view(kp, page, p % ps, h), want_k):
                        bad.append(f"K row of token {t} wrong")
                    if not np.array_equal(view(vp, page, p % ps, h), v[t, h]):
                        bad.append(f"V row of token {t} wrong")
            for page in range(num_pages):
                for slot in range(ps):
                    for h in range(Hkv):
                        if (page, slot, h) in changed:
                            continue
                        if not (np.array_equal(view(kp, page, slot, h), view(k_pages, page, slot, h))
                                and np.array_equal(view(vp, page, slot, h),
                                                   view(v_pages, page, slot, h))):
                            bad.append(f"untouched row ({page}, {slot}, {h}) changed")
    return bad


# ------------------------------------------------------------------ tests

def test_rope_pins():
    assert rope_pins(None) == []


def test_append_pins():
    assert append_pins(None) == []


def test_bf16_pins():
    assert bf16_pins(None) == []


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(2000).astype(np.float32),
                        np.float32([1.0, 1.00390625, 1.005859375, -2.00781250, 65504.0, 1e-3])])
    want = torch.as_tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(x.astype(np.float64)), want)


ROPE_MUTANTS = {
    "interleaved_pairs": ("yr[i] = xr[i] * c - xr[i + h] * s;\n            yr[i + h] = xr[i + h] * c + xr[i] * s;",
                          "yr[2 * i] = xr[2 * i] * c - xr[2 * i + 1] * s;\n            yr[2 * i + 1] = xr[2 * i + 1] * c + xr[2 * i] * s;"),
    "sine_sign": ("yr[i] = xr[i] * c - xr[i + h] * s;", "yr[i] = xr[i] * c + xr[i + h] * s;"),
    "frequency_exponent": ("const double f = pow(theta, -2.0 * (double)i / (double)D);",
                           "const double f = pow(theta, -(double)i / (double)D);"),
    "slot_from_page": ("const int slot = p % page_size;", "const int slot = (p + 1) % page_size;"),
    "ignores_refcount": ("else if (refcount[page] != 1)", "else if (refcount[page] < 1)"),
    # converting to f32 before rounding to bf16 rounds twice
    "bf16_through_f32": ("const double m = frexp(x, &e);           /* x = m * 2^e, 0.5 <= |m| < 1 */",
                         "const double m = frexp((double)(float)x, &e);"),
    "bf16_subnormal_truncated": ("r = ldexp(nearbyint(ldexp(x, 133)), -133);",
                                 "r = ldexp(trunc(ldexp(x, 133)), -133);"),
    "bf16_no_subnormal_step": ("} else if (fabs(x) < ldexp(1.0, -126)) {", "} else if (0) {"),
    "pool_past_last_page": (
        "(int64_t)p >= ((int64_t)indptr[b + 1] - indptr[b]) * (int64_t)page_size) {",
        "(int64_t)p > ((int64_t)indptr[b + 1] - indptr[b]) * (int64_t)page_size) {"),
}


@pytest.mark.parametrize("name", sorted(ROPE_MUTANTS))
def test_pins_reject_planted_mistakes(name, tmp_path):
    old, new = ROPE_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mutated = tmp_path / "oxd_oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oxd_oracle.h").write_text(open(SRC[:-1] + "h").read())
    lib = oracle.bind(oracle.compile_library(str(mutated), str(tmp_path / f"lib_{name}.so")))
    try:
        failures = rope_pins(lib) + append_pins(lib) + bf16_pins(lib)
    except Exception as e:  # a mutant may also crash the battery
        failures = [repr(e)]
    assert failures, f"mutant {name} passed every pin"
