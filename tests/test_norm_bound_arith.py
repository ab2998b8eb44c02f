"""The arithmetic behind the six-bit shortcut of the fused kernel, checked on
the CPU against the oracle's MX scale rule.

With six-bit P (MXFP6, MXFP4) a 32-key block whose largest bf16 weight code
is C gets the E2M3 scale 2^X by the scale rule (smallest X with
p_max <= 7.5 * 2^X), and the kernel stores p / 2^(X+6) as an E4M3 pattern.
Its scaled conversion is exact for a code c when c >= 128 (a normal bf16)
and c >= 128 (X + 7) (p / 2^(X+6) a normal FP32 whose pattern is
(c << 16) - ((X + 6) << 23)).  The kernel skips the block minima for a warp
when 2 |alpha| A <= 15000 (A = |q^_i| max_j |k^_j|); this holds when every
code of the tile is within 15601 of the tile's largest and at least 128,
which is what these tests pin, for every bf16 code."""
import oracle

LIMIT = 15000.0  # the kernel's bound on 2 |alpha| A
SPAN = 15601     # largest code distance the scaled conversion tolerates
ROUND = 0.51     # codes lie within this of alpha (acc - m) + 16249


def test_span_covers_the_scale_rule_for_every_code():
    for C in range(0, 0x7F80):  # every finite non-negative bf16 weight code
        p_max = oracle.bf16_to_double(C)
        X = oracle.mx_scale_exp(oracle.E2M3, p_max)
        need = max(128, 128 * (X + 7))  # smallest code the scaled conversion takes
        allowed = max(128, C - SPAN)    # smallest code the bound guarantees
        assert need <= allowed, (C, X)


def test_span_is_tight():
    # one code more of distance would break the rule for some block maximum
    worst = min(max(128, C - (SPAN + 1)) - max(128, 128 * (oracle.mx_scale_exp(oracle.E2M3, oracle.bf16_to_double(C)) + 7))
                for C in range(0, 0x7F80))
    assert worst < 0


def test_limit_leaves_room_for_rounding():
    # spread: C - c_min <= 2 |alpha| A + 2 ROUND; floor: c_min >= 16249 - 2 |alpha| A - ROUND
    assert LIMIT + 2 * ROUND <= SPAN
    assert 16249 - LIMIT - ROUND >= 128
    # the margin left for the tensor core's accumulation error, relative
    assert (SPAN - 2 * ROUND) / LIMIT - 1 > 0.03
