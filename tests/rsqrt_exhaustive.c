/* Checks that RN32(1.0 / sqrt((double)v)) -- the oracle's rrms step -- is the correctly rounded
 * fp32 reciprocal square root for positive finite fp32 bit patterns u in [lo, hi) stepping by
 * `step`. The neighbours' midpoints m have at most 25 significant bits, so m*m is exact in
 * binary64 and the sign of fma(m*m, v, -1) (one rounding of an exact product) decides on which
 * side of 1/sqrt(v) each midpoint lies. Prints "checked N mismatches M"; exit status 1 on any
 * mismatch. Test support for tests/test_oracle_pins.py (the default run samples the range). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

int main(int argc, char** argv) {
    uint32_t lo = argc > 1 ? (uint32_t)strtoul(argv[1], 0, 0) : 1u;
    uint32_t hi = argc > 2 ? (uint32_t)strtoul(argv[2], 0, 0) : 0x7f800000u;
    uint32_t step = argc > 3 ? (uint32_t)strtoul(argv[3], 0, 0) : 1u;
    unsigned long long n = 0, bad = 0;
    for (uint64_t w = lo; w < hi; w += step) {
        uint32_t u = (uint32_t)w;
        float v;
        memcpy(&v, &u, 4);
        float y = (float)(1.0 / sqrt((double)v));
        float up = nextafterf(y, INFINITY), dn = nextafterf(y, 0.0f);
        double mu = ((double)y + (double)up) * 0.5, md = ((double)y + (double)dn) * 0.5;
        /* correct rounding: md < 1/sqrt(v) < mu, i.e. md^2 v < 1 < mu^2 v */
        if (!(fma(mu * mu, (double)v, -1.0) > 0.0 && fma(md * md, (double)v, -1.0) < 0.0)) {
            if (bad < 5) printf("mismatch at %08x\n", u);
            ++bad;
        }
        ++n;
    }
    printf("checked %llu mismatches %llu\n", n, bad);
    return bad != 0;
}
