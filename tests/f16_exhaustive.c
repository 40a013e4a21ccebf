/* Exhaustive check of the oracle's binary32 -> binary16 rounding against the
 * C compiler's _Float16 conversion (a library routine: libgcc's
 * __truncsfhf2 on x86-64, the FCVT instruction on AArch64), over all 2^32
 * binary32 bit patterns.  NaNs must map to NaNs (payloads may differ).
 * Prints the mismatch count; exit status 0 when it is zero. */
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

uint16_t oracle_f32_to_f16_rn(float v);

#define NT 16
static uint64_t bad[NT];
static uint32_t first_bad[NT];

static void* run(void* arg)
{
    int t = (int)(intptr_t)arg;
    uint64_t lo = ((uint64_t)1 << 32) / NT * t, hi = ((uint64_t)1 << 32) / NT * (t + 1);
    for (uint64_t i = lo; i < hi; ++i) {
        uint32_t u = (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        uint16_t mine = oracle_f32_to_f16_rn(f);
        _Float16 h = (_Float16)f;
        uint16_t ref;
        memcpy(&ref, &h, 2);
        int nan_in = ((u >> 23) & 0xff) == 0xff && (u & 0x7fffff);
        int ok;
        if (nan_in)
            ok = ((mine & 0x7c00) == 0x7c00) && (mine & 0x3ff) && ((mine ^ (u >> 16)) & 0x8000) == 0;
        else
            ok = mine == ref;
        if (!ok) { if (!bad[t]) first_bad[t] = u; ++bad[t]; }
    }
    return 0;
}

int main(void)
{
    pthread_t th[NT];
    for (int t = 0; t < NT; ++t) pthread_create(&th[t], 0, run, (void*)(intptr_t)t);
    uint64_t total = 0;
    for (int t = 0; t < NT; ++t) {
        pthread_join(th[t], 0);
        if (bad[t]) printf("first mismatch in slice %d: 0x%08x\n", t, first_bad[t]);
        total += bad[t];
    }
    printf("mismatches %llu\n", (unsigned long long)total);
    return total != 0;
}
