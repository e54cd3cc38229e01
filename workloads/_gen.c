/* Host side of the counter-based bf16 generator in workloads/__init__.py.
 *
 * out[i] = table[hash(start + i) >> 16], hash = mix32(mix32(idx * C0 ^ k1) ^ k2).
 * Bit-identical to the numpy and torch formulations of the same hash.
 * Holds no arithmetic of the decoder itself.
 */
#include <stdint.h>

static inline uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x5BD1E995u;
    x ^= x >> 16;
    return x;
}

static inline uint32_t hash_idx(uint32_t idx, uint32_t k1, uint32_t k2) {
    return mix32(mix32(idx * 0x61C88647u ^ k1) ^ k2);
}

void gen_bf16(uint32_t k1, uint32_t k2, const uint16_t *table,
              uint64_t start, uint64_t n, uint16_t *out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; ++i)
        out[i] = table[hash_idx((uint32_t)(start + (uint64_t)i), k1, k2) >> 16];
}

void gen_bf16_rows(uint32_t k1, uint32_t k2, const uint16_t *table,
                   const int64_t *rows, int64_t nrows, int64_t ncol, uint16_t *out) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t c = 0; c < ncol; ++c)
            out[r * ncol + c] = table[hash_idx((uint32_t)(rows[r] * ncol + c), k1, k2) >> 16];
}
