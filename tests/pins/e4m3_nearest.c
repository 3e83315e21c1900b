/*
 * Independent pin for the oracle's fp32 -> E4M3 encoder, used by the CPU
 * tests only.  It does not reuse the oracle's method (binade + quantum +
 * nearbyint): it lists the 127 non-negative finite E4M3 values, which rise
 * with the code, and finds the nearest one by binary search.  A tie goes to
 * the even code; anything at or above 448 (inf included) saturates to 448.
 * The sign is copied from the input, NaN inputs are skipped.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

static double table[127];

static void fill_table(void) {
    /* code c = eeee.mmm (no sign): the value doubles every 8 codes from
     * 2^-6 upward; the first 8 codes step by 2^-9 from zero. */
    for (int c = 0; c < 127; ++c) {
        if (c < 8) table[c] = c / 512.0;
        else {
            double base = 1.0 / 64.0;            /* code 8 */
            for (int b = 8; b + 8 <= c; b += 8) base *= 2.0;
            table[c] = base * (1.0 + (c & 7) / 8.0);
        }
    }
}

static uint8_t nearest(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 126;
    int lo = 0, hi = 126;                      /* table[lo] <= a < table[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (table[mid] <= a) lo = mid; else hi = mid;
    }
    double dl = a - table[lo], dh = table[hi] - a;
    int c = (dl < dh) ? lo : (dh < dl) ? hi : ((lo % 2 == 0) ? lo : hi);
    return sign | (uint8_t)c;
}

/* Compare q[i] (the oracle's code for bit pattern start+i) with the nearest
 * search; return the mismatch count and the first mismatching index. */
int64_t check_chunk(uint64_t start, int64_t n, const uint8_t* q, int64_t* first_bad) {
    static int ready = 0;
    if (!ready) { fill_table(); ready = 1; }
    int64_t bad = 0, first = -1;
#pragma omp parallel for reduction(+:bad) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)(start + (uint64_t)i);
        float f;
        memcpy(&f, &u, sizeof f);
        if (isnan(f)) continue;
        if (nearest(f) != q[i]) {
            bad++;
#pragma omp critical
            if (first < 0 || i < first) first = i;
        }
    }
    *first_bad = first;
    return bad;
}

double table_value(int c) {
    fill_table();
    return table[c];
}
