/* synth_host.c -- host C twin of synth/gen.py's counter-based normal
 * generator (SplitMix64 output function, Irwin-Hall(12) normals, bf16 RNE),
 * for filling large host arrays quickly.  Input generation only. */
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint16_t normal_bf16_at(uint64_t key, uint64_t idx)
{
    int64_t s = 0;
    const uint64_t c0 = idx * 3ull;
    for (int j = 0; j < 3; ++j) {
        const uint64_t h = mix64(key + (c0 + (uint64_t)j + 1ull) * 0x9E3779B97F4A7C15ull);
        for (int k = 0; k < 4; ++k)
            s += (int64_t)((h >> (16 * k)) & 0xFFFFull);
    }
    /* (S - 393210) is exact in fp32 and the scaling by 2^-16 is exact */
    const float x = (float)(s - 393210) * (1.0f / 65536.0f);
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* out[i] = bf16 normal at counter idx[i] */
void synth_normal_bf16_idx(uint16_t *out, uint64_t key, const uint64_t *idx, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = normal_bf16_at(key, idx[i]);
}

/* out[i] = bf16 normal at counter base + i */
void synth_normal_bf16_range(uint16_t *out, uint64_t key, uint64_t base, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = normal_bf16_at(key, base + (uint64_t)i);
}

/* rows of row_len contiguous counters starting at base + r * row_stride */
void synth_normal_bf16_rows(uint16_t *out, uint64_t key, uint64_t base, int64_t rows, int64_t row_len,
                            uint64_t row_stride)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < row_len; ++i)
            out[r * row_len + i] = normal_bf16_at(key, base + (uint64_t)r * row_stride + (uint64_t)i);
}
