/* Independent reference rounding float -> bf16 for the oracle's exhaustive pin.
 * Bracket-and-compare: the two bf16 neighbours of f are the truncated pattern
 * and the next pattern away from zero; pick the nearer by comparing exact
 * distances in double, and on a tie the one whose last kept bit is 0.
 * NaN inputs map to 0xFFFF (the test checks them separately). */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double val(uint32_t bits) { float f; memcpy(&f, &bits, 4); return (double)f; }

void bracket_range(uint64_t lo_u, uint64_t hi_u, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = (int64_t)lo_u; i < (int64_t)hi_u; ++i) {
        uint32_t u = (uint32_t)i;
        double f = val(u);
        uint16_t r;
        if (isnan(f)) r = 0xFFFFu;
        else if (isinf(f)) r = (uint16_t)(u >> 16);
        else {
            uint32_t down = u & 0xFFFF0000u, up = down + 0x10000u;
            double dd = fabs(f - val(down));
            double du = isinf(val(up)) ? fabs(ldexp(1.0, 128) - fabs(f)) : fabs(val(up) - f);
            if (dd < du) r = (uint16_t)(down >> 16);
            else if (du < dd) r = (uint16_t)(up >> 16);
            else r = ((down >> 16) & 1u) ? (uint16_t)(up >> 16) : (uint16_t)(down >> 16);
        }
        out[i - (int64_t)lo_u] = r;
    }
}
