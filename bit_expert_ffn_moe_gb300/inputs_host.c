/* Host implementation of the counter-based SplitMix64 weight generator of inputs.py (input
 * generation only; none of the layer's arithmetic).  Element n of the stream with key `key` is
 * float32(2*(u0+u1+u2+u3) - 262140) * c, u0..u3 the 16-bit fields of mix(key + (n+1)*golden). */
#include <stdint.h>

static uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t inputs_stream_key(uint64_t seed, uint32_t tensor_id, uint32_t expert) {
    return mix((seed << 32) | ((uint64_t)tensor_id << 24) | (uint64_t)expert);
}

void inputs_synth(uint64_t key, int64_t first, int64_t n, float c, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t z = mix(key + (uint64_t)(first + i + 1) * 0x9E3779B97F4A7C15ull);
        int32_t s = (int32_t)(z & 0xFFFF) + (int32_t)((z >> 16) & 0xFFFF) + (int32_t)((z >> 32) & 0xFFFF) +
                    (int32_t)((z >> 48) & 0xFFFF);
        volatile float v = (float)(2 * s - 262140);
        out[i] = v * c;
    }
}
