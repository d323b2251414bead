"""The FP8 kernels divide x by the block scale s without a division: with
y = RN(1/s), q0 = RN(x y), then twice r = RN(s q - x), q = RN(q - r y)
(Markstein's correction with the residual formed negated, so that x = -0
keeps a -0 quotient). This checks the sequence on the host against the IEEE
quotient RN(x / s) for scales across [2^-90, 2^90] and values up to the
block maximum 448 s: bit-identical wherever |x / s| >= 2^-11 (every quotient
that can reach a non-zero E4M3 code), and a quotient of the sign of x no
larger than 2^-10 in magnitude below that (which rounds to a zero code of
that sign, as the division's does). The reference quotient and reciprocal are
binary64 operations rounded to binary32, exact here: for binary32 operands a
binary64 intermediate makes double rounding of a quotient innocuous
(Figueroa, "When is double rounding innocuous?", SIGNUM Newsletter 30(3),
1995)."""
import subprocess
import tempfile
from pathlib import Path

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static uint64_t st = 0x9E3779B97F4A7C15ull;
static uint64_t next(void) {  /* SplitMix64 */
    uint64_t z = (st += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float quotient(float x, float s) {
    const float y = (float)(1.0 / (double)s);
    float q = x * y;
    float r = fmaf(s, q, -x);
    q = fmaf(r, -y, q);
    r = fmaf(s, q, -x);
    return fmaf(r, -y, q);
}

int main(int argc, char **argv) {
    const long n = strtol(argv[1], 0, 10);
    long bad = 0, exact = 0, small = 0;
    for (long i = 0; i < n; ++i) {
        /* s: a random binary32 in [2^-90, 2^90] */
        const uint32_t slo = 0x1A800000u, shi = 0x66800000u;
        const float s = f_of(slo + (uint32_t)(next() % (uint64_t)(shi - slo + 1)));
        const float amax = (float)((double)s * 448.0);
        float x;
        const uint64_t kind = next() % 8;
        if (kind == 0) x = 0.0f;
        else if (kind == 1) x = -0.0f;
        else if (kind == 2) x = f_of((uint32_t)(next() % 0x00800000u));  /* subnormal */
        else if (kind == 3) x = amax;
        else if (kind == 4) x = f_of((uint32_t)(next() % (u_of(amax) + 1)));  /* any magnitude up to amax */
        else x = (float)((double)amax * (double)(next() >> 11) * 0x1p-53);  /* uniform in [0, amax) */
        if (next() & 1) x = -x;
        const float want = (float)((double)x / (double)s), got = quotient(x, s);
        if (fabs((double)x / (double)s) >= 0x1p-11) {
            ++exact;
            if (u_of(want) != u_of(got)) ++bad;
        } else {
            ++small;
            if (signbit(got) != signbit(x) || fabsf(got) > 0x1p-10f) ++bad;
        }
    }
    printf("%ld %ld %ld\n", exact, small, bad);
    return 0;
}
"""


def test_division_free_quotient_equals_the_ieee_quotient():
    with tempfile.TemporaryDirectory() as d:
        c, exe = Path(d) / "q.c", Path(d) / "q"
        c.write_text(SRC)
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", str(c), "-o", str(exe), "-lm"], check=True)
        out = subprocess.run([str(exe), "4000000"], check=True, capture_output=True, text=True).stdout.split()
    exact, small, bad = (int(v) for v in out)
    assert exact > 2_000_000 and small > 100_000
    assert bad == 0
