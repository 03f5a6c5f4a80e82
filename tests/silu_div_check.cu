// Checks the SiLU quotient of the L1 epilogue (div_by_ge1, Markstein's method)
// against the division operator, bit for bit:
//   1. every BF16 value g (the epilogue rounds the accumulator to BF16 before
//      SiLU): g / (1 + expf(-g));
//   2. 2^24 pseudo-random float pairs: a any float (specials included), b in
//      [1, 2^128) or, for every 4096th pair, +inf; pairs with 0 < |a| < 2^-100
//      or a subnormal quotient are not counted (they may differ in the last
//      place).
// The packed two-quotient form (div_by_ge1x2) is held to the same bars: in
// both checks its halves must equal the scalar form.
// Prints "mismatches <n1> <n2>" and exits 0 if the kernels ran.
#include "common.cuh"

#include <cstdio>
#include <cstring>

using moeffn::div_by_ge1;
using moeffn::div_by_ge1x2;

__device__ __forceinline__ bool same_bits(float x, float y) {
    return (isnan(x) && isnan(y)) || __float_as_uint(x) == __float_as_uint(y);
}

__global__ void check_bf16(unsigned int* bad, float* rec) {
    const unsigned int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 65536u) return;
    const float g = __uint_as_float(i << 16);
    const float b = 1.0f + expf(-g);
    const float q = div_by_ge1(g, b), r = g / b;
    // the packed form, this value in either half (the other half: the next BF16 value)
    const float g2 = __uint_as_float(((i + 1u) & 0xFFFFu) << 16);
    const float2 p = div_by_ge1x2(make_float2(g, g2), make_float2(b, 1.0f + expf(-g2)));
    const float2 p2 = div_by_ge1x2(make_float2(g2, g), make_float2(1.0f + expf(-g2), b));
    if (!same_bits(q, r) || !same_bits(p.x, r) || !same_bits(p2.y, r)) {
        const unsigned int k = atomicAdd(bad, 1u);
        if (k < 8) { rec[4 * k] = g; rec[4 * k + 1] = b; rec[4 * k + 2] = q; rec[4 * k + 3] = r; }
    }
}

__device__ __forceinline__ unsigned int mix(unsigned int x) {   // a 32-bit integer hash
    x ^= x >> 16; x *= 0x7feb352du; x ^= x >> 15; x *= 0x846ca68bu; x ^= x >> 16;
    return x;
}

__global__ void check_random(unsigned int n, unsigned int* bad, float* rec) {
    const unsigned int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const unsigned int ra = mix(2u * i + 1u), rb = mix(2u * i + 2u);
    const float a = __uint_as_float(ra);                       // any float, specials included
    // b in [1, 2^127]: exponent 127..254, any mantissa; every 4096th: +inf
    float b = __uint_as_float(((127u + rb % 128u) << 23) | (mix(rb) & 0x7FFFFFu));
    if ((i & 4095u) == 0) b = __uint_as_float(0x7F800000u);
    const float q = div_by_ge1(a, b), r = a / b;
    // the packed form with this pair in either half must equal the scalar form everywhere
    const float2 p1 = div_by_ge1x2(make_float2(a, 1.0f), make_float2(b, 3.0f));
    const float2 p2 = div_by_ge1x2(make_float2(-1.0f, a), make_float2(2.0f, b));
    const bool packed_ok = same_bits(p1.x, q) && same_bits(p2.y, q);
    // a dividend below 2^-100 in magnitude (or a subnormal quotient) may differ in
    // the last place; the exhaustive check above covers every BF16 input of SiLU
    const bool tiny = (a != 0.0f && fabsf(a) < 0x1p-100f) || (r != 0.0f && fabsf(r) < 0x1p-126f);
    if ((!tiny && !same_bits(q, r)) || !packed_ok) {
        const unsigned int k = atomicAdd(bad, 1u);
        if (k < 8) { rec[4 * k] = a; rec[4 * k + 1] = b; rec[4 * k + 2] = q; rec[4 * k + 3] = r; }
    }
}

int main() {
    unsigned int* d;
    float* rec;
    if (cudaMalloc(&d, 8) != cudaSuccess || cudaMalloc(&rec, 2 * 32 * sizeof(float)) != cudaSuccess) return 2;
    cudaMemset(d, 0, 8);
    check_bf16<<<256, 256>>>(d, rec);
    const unsigned int n = 1u << 24;
    check_random<<<(n + 255) / 256, 256>>>(n, d + 1, rec + 32);
    if (cudaDeviceSynchronize() != cudaSuccess) return 3;
    unsigned int h[2];
    float hr[64];
    cudaMemcpy(h, d, 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(hr, rec, sizeof(hr), cudaMemcpyDeviceToHost);
    std::printf("mismatches %u %u\n", h[0], h[1]);
    for (int c = 0; c < 2; ++c)
        for (unsigned int k = 0; k < h[c] && k < 8; ++k) {
            const float* r = hr + 32 * c + 4 * k;
            unsigned int u[4];
            std::memcpy(u, r, 16);
            std::printf("  %s a %a b %a got %a (%08x) want %a (%08x)\n", c ? "random" : "bf16", r[0], r[1], r[2], u[2],
                        r[3], u[3]);
        }
    return 0;
}
