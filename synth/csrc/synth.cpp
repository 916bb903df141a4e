// Native twin of the ternary draw in synth/__init__.py, for regenerating the
// 52-billion-weight c2048-shaped layer quickly.  It draws random numbers and
// nothing else.  Same definition: SplitMix64 in counter mode, weight (r, c)
// uses stream index r*cols + c of the stream keyed by
// splitmix64(seed, (1 << 48) | (expert << 8) | matrix); zero when the high 32
// bits of the draw are below `threshold`, else +1 for an odd draw, -1 for an
// even one.
#include <cstdint>

namespace {
inline uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
inline uint64_t at(uint64_t key, uint64_t idx) { return mix(key + (idx + 1) * 0x9E3779B97F4A7C15ull); }
}  // namespace

extern "C" void synth_ternary_rows(uint64_t seed, uint32_t expert, uint32_t matrix, int64_t cols,
                                   uint32_t threshold, int64_t row_start, int64_t row_count, int8_t* out) {
    const uint64_t key = at(seed, ((uint64_t)1 << 48) | ((uint64_t)expert << 8) | (uint64_t)matrix);
    for (int64_t r = 0; r < row_count; ++r) {
        const uint64_t base = (uint64_t)(row_start + r) * (uint64_t)cols;
        int8_t* o = out + r * cols;
        for (int64_t c = 0; c < cols; ++c) {
            const uint64_t u = at(key, base + (uint64_t)c);
            const int8_t sgn = (int8_t)(((int)(u & 1u) << 1) - 1);     // +1 odd, -1 even
            const int8_t nz = (int8_t)((uint32_t)(u >> 32) >= threshold);
            o[c] = (int8_t)(sgn * nz);
        }
    }
}
