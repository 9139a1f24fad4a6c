"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that a pin catches each one: the pins constrain every layer of the oracle,
not just its overall statistics."""
import pytest

import oracle
import pins

# (name, text in oracle.c, replacement, pin that must fail)
MUTATIONS = [
    ("hash shift 15->16", "x = mix(x, 15);", "x = mix(x, 16);", pins.pin_tile_mean),
    ("hash multiplier", "x = x * 2146121005u;", "x = x * 2146121007u;", pins.pin_tile_mean),
    ("unhashed seed key", "return orc_hash32(counter ^ orc_hash32(seed));",
     "return orc_hash32(counter ^ seed);", pins.pin_tile_mean),
    ("arithmetic shift", "return x ^ (x >> s); }", "return x ^ (uint32_t)((int32_t)x >> s); }",
     pins.pin_tile_mean),
    ("24-bit uniform mask", "& 8388607u) * 1.1920928955078125e-7f",
     "& 16777215u) * 1.1920928955078125e-7f", pins.pin_tile_mean),
    ("u8 byte order", "return (uint8_t)(orc_draw32(seed, counter >> 2) >> (8u * (counter & 3u)));",
     "return (uint8_t)(orc_draw32(seed, counter >> 2) >> (8u * (3u - (counter & 3u))));", pins.pin_narrow_fills),
    ("bool bit index", "return (uint8_t)((orc_draw32(seed, counter >> 5) >> (counter & 31u)) & 1u);",
     "return (uint8_t)((orc_draw32(seed, counter >> 5) >> (31u - (counter & 31u))) & 1u);", pins.pin_narrow_fills),
    ("f16 exponent", "return (uint16_t)(((p + 5u) << 10) | fraction);", "return (uint16_t)(((p + 6u) << 10) | fraction);",
     pins.pin_narrow_fills),
    ("64-bit word order",
     "return ((uint64_t)orc_draw32(seed, c2) << 32) | (uint64_t)orc_draw32(seed, c2 + 1u);",
     "return ((uint64_t)orc_draw32(seed, c2 + 1u) << 32) | (uint64_t)orc_draw32(seed, c2);",
     pins.pin_draw64_words),
    ("f64 takes 52 bits", "return (double)(orc_draw64(seed, counter) >> 11) * 0x1p-53;",
     "return (double)(orc_draw64(seed, counter) >> 12) * 0x1p-53;", pins.pin_draw64_words),
    ("Lemire strict compare", "return low >= threshold;", "return low > threshold;",
     pins.pin_lemire_exhaustive_8bit),
    ("Lemire threshold", "uint64_t threshold = (uint64_t)(two_w % b);",
     "uint64_t threshold = (uint64_t)((two_w - 1) % b);", pins.pin_lemire_exhaustive_8bit),
    ("Lemire modulo value", "*value = (uint64_t)(prod / two_w);", "*value = x % b;",
     pins.pin_lemire_exhaustive_8bit),
    ("range without low", "return (int32_t)((uint32_t)low + orc_below32(seed, counter, b));",
     "return (int32_t)orc_below32(seed, counter, b);", pins.pin_ranges_wrap),
    ("randn sin branch", "return sqrt(-2.0 * log(1.0 - u0)) * cos(6.283185307179586 * u1);",
     "return sqrt(-2.0 * log(1.0 - u0)) * sin(6.283185307179586 * u1);", pins.pin_randn_special_angles),
    ("randn half turn", "return sqrt(-2.0 * log(1.0 - u0)) * cos(6.283185307179586 * u1);",
     "return sqrt(-2.0 * log(1.0 - u0)) * cos(3.141592653589793 * u1);", pins.pin_randn_special_angles),
    ("randn swapped counters",
     "double u0 = (double)orc_uniform_f32(seed, 2u * counter);",
     "double u0 = (double)orc_uniform_f32(seed, 2u * counter + 1u);",
     pins.pin_randn_special_angles),
    ("randn log(u)", "return sqrt(-2.0 * log(1.0 - u0)) * cos(6.283185307179586 * u1);",
     "return sqrt(-2.0 * log(u0 + 0x1p-24)) * cos(6.283185307179586 * u1);", pins.pin_randn_special_angles),
    ("paired sine for cosine", "return (counter & 1u) ? r * sin(6.283185307179586 * u1) : r * cos(6.283185307179586 * u1);",
     "return (counter & 1u) ? r * cos(6.283185307179586 * u1) : r * sin(6.283185307179586 * u1);",
     pins.pin_randn_paired),
    ("paired pair index", "    uint32_t q = counter >> 1;", "    uint32_t q = (counter + 1u) >> 1;", pins.pin_randn_paired),
    ("exponential f32 of u", "return -log(1.0 - (double)orc_uniform_f32(seed, counter));",
     "return -log((double)orc_uniform_f32(seed, counter) + 0x1p-24);", pins.pin_exponentials),
    ("exponential f64 sign", "return 0.0 - orc_zlog(v);", "return orc_zlog(v);", pins.pin_exponentials),
    ("dropout drops ties", "return (u >= p) ? x / keep_scale_divisor : 0.0f;",
     "return (u > p) ? x / keep_scale_divisor : 0.0f;", pins.pin_dropout),
    ("dropout reciprocal multiply", "return (u >= p) ? x / keep_scale_divisor : 0.0f;",
     "return (u >= p) ? x * (1.0f / keep_scale_divisor) : 0.0f;", pins.pin_dropout),
    ("dropout no rescale", "return (u >= p) ? x / keep_scale_divisor : 0.0f;",
     "return (u >= p) ? x : 0.0f;", pins.pin_dropout),
    ("zexp dropped term", "p = fma(p, r, 1.0 / 720.0);       /* 1/6! */",
     "p = fma(p, r, 0.0);", pins.pin_zexp_zlog),
    ("zlog exponent sign", "e = e + 1;", "e = e - 1;", pins.pin_zexp_zlog),
    ("zlog missing series term", "p = fma(p, s2, 1.0 / 3.0);", "p = fma(p, s2, 0.0);",
     pins.pin_zexp_zlog),
    ("ziggurat tail area dropped", "return r * qf(r) + Q_SQRT(pi / 2) * Q_ERFC(r / Q_SQRT((quad)2));",
     "return r * qf(r);", pins.pin_zig_table_published),
    ("ziggurat base width", "X[0] = (double)(v / qf(r));", "X[0] = (double)(r);",
     pins.pin_zig_table_invariants),
    ("ziggurat fast test", "return x < zig_X[j + 1];", "return x < zig_X[j];",
     pins.pin_zig_miss_rate),
    ("ziggurat wedge compare", "if (y < orc_zexp(t)) return neg ? -x : x;",
     "if (y > orc_zexp(t)) return neg ? -x : x;", pins.pin_zig_wedge_acceptance),
    ("ziggurat wedge interpolation", "double y = zig_F[j] + u * (zig_F[j + 1] - zig_F[j]);",
     "double y = zig_F[j] + u * (zig_F[j + 1] - zig_F[j]) * 0.5;", pins.pin_zig_wedge_acceptance),
    ("ziggurat sign bit", "int neg = (int)((w >> 10) & 1u);", "int neg = (int)((w >> 11) & 1u);",
     pins.pin_zig_wedge_acceptance),
    ("ziggurat tail sign", "double z = r + a;", "double z = r - a;",
     pins.pin_normal_f64_distribution),
    ("ziggurat tail scale", "double a = -orc_zlog(u1) / r;", "double a = -orc_zlog(u1);",
     pins.pin_normal_f64_distribution),
]


@pytest.mark.parametrize("name,old,new,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_mutation(tmp_path, name, old, new, pin):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    mutant = oracle.variant(src.replace(old, new), str(tmp_path))
    with pytest.raises(AssertionError):
        pin(mutant)
