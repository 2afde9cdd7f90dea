/* The FP8 codec's division method, restated in plain C for a check against
 * IEEE fp32 division.  The CUDA codec divides x by the block scale s through
 * y = RN(1/s): q0 = RN(x*y), r = RN(q0*s - x) (one fma, exact), then
 * q = RN(q0 - r*y) (one fma) -- Markstein's correction step -- for scales in
 * [2^-100, 3e38]; other scales use the IEEE division itself.  This program
 * walks block maxima a (bf16 bit patterns first, first+stride, ... up to last,
 * by default the largest finite bf16), sets s = RN(a / 448), and for every bf16 x with
 * |x| <= a (and every NaN x) compares the e4m3 code of q with the code of the
 * IEEE quotient x / s, using the oracle's encoder.  Prints "pairs mismatches
 * quotient_mismatches_at_or_above_2^-10" and exits 1 on any code mismatch.
 * Build with -ffp-contract=off so that x*y is rounded on its own. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ep_oracle.h"

static float from_bf16(uint32_t b) {
    uint32_t u = b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t bits_of(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

int main(int argc, char** argv) {
    const uint32_t first = argc > 1 ? (uint32_t)atoi(argv[1]) : 1;
    const uint32_t stride = argc > 2 ? (uint32_t)atoi(argv[2]) : 1;
    const uint32_t last = argc > 3 ? (uint32_t)atoi(argv[3]) : 0x7F7Fu;
    long long pairs = 0, bad_code = 0, bad_quot = 0;
    for (uint32_t ab = first; ab <= last && ab <= 0x7F7Fu; ab += stride) {
        const float amax = from_bf16(ab);
        volatile float sv = amax / 448.0f;
        const float s = sv;
        if (!(s >= 0x1p-100f && s <= 3.0e38f)) continue;
        volatile float yv = 1.0f / s;
        const float y = yv;
        for (uint32_t xb = 0; xb < 0x10000u; ++xb) {
            const float x = from_bf16(xb);
            if (!(fabsf(x) <= amax) && !isnan(x)) continue;
            volatile float q0v = x * y;
            const float q0 = q0v;
            const float r = fmaf(q0, s, -x);
            const float q = fmaf(-r, y, q0);
            const float ref = x / s;
            ++pairs;
            const uint8_t cq = orc_e4m3_encode(q), cr = orc_e4m3_encode(ref);
            const int same = isnan(x) ? ((cq & 0x7F) == 0x7F && (cr & 0x7F) == 0x7F) : (cq == cr);
            if (!same) {
                if (bad_code < 5) fprintf(stderr, "amax %a x %a: code %02x, IEEE %02x\n", amax, x, cq, cr);
                ++bad_code;
            }
            if (!isnan(x) && bits_of(q) != bits_of(ref) && fabsf(ref) >= 0x1p-10f) ++bad_quot;
        }
    }
    printf("%lld %lld %lld\n", pairs, bad_code, bad_quot);
    return bad_code ? 1 : 0;
}
