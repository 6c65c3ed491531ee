// fp8.cu -- FP8 (E4M3) block quantisation: static quantisation of the expert weights in
// 128 x 128 tiles and the dynamic quantise-dequantise of activation rows in vectors of
// 128, both with power-of-two scales.
//
// Method: "Lower latency and higher throughput with multi-node DeepSeek deployment",
// section "Quantization": weights are quantised ahead of time with one scale per 128 x 128
// tile, activations on the fly with one scale per 128-element vector.  Scale of a block:
// the smallest 2^k with amax <= 448 * 2^k (E4M3's largest finite value is 448), k within
// [-124, 127]; q = E4M3 round-to-nearest-even of x / 2^k.  The expert FFN multiplies the
// E4M3 bytes on the tensor cores (one 128-wide block of the reduction at a time) and
// applies the two blocks' scales to each block's fp32 partial sum.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int QB = 128;   // block edge

// One CTA per 128 x 128 tile of W[g] ([R][C], R the reduction dimension): 256 threads,
// each a 64-element half row.  The E4M3 bytes are written transposed, Wq[g][C][R] (each
// output column's R values contiguous: the K-major operand rows the FP8 tensor-core MMA
// reads), through a shared-memory tile.
__global__ void __launch_bounds__(256) quant_weight_kernel(const uint16_t *__restrict__ W, int R,
                                                           int C, uint8_t *__restrict__ Wq,
                                                           int32_t *__restrict__ S)
{
    pdl_wait();
    __shared__ float red[8];
    __shared__ __align__(16) uint8_t tile[QB][QB + 16];   // [c][r], padded rows
    const int cb = blockIdx.x, rb = blockIdx.y, g = blockIdx.z;
    const int t = threadIdx.x, rl = t >> 1, cl0 = (t & 1) * 64;
    const int r = rb * QB + rl, c0 = cb * QB + cl0;
    const size_t off = (static_cast<size_t>(g) * R + r) * C + c0;
    const uint4 *src = reinterpret_cast<const uint4 *>(W + off);
    float v[64];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 u = __ldg(src + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = bf16_lo(w[j]);
            v[8 * i + 2 * j + 1] = bf16_hi(w[j]);
            amax = fmaxf(amax, fmaxf(fabsf(v[8 * i + 2 * j]), fabsf(v[8 * i + 2 * j + 1])));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
    if ((t & 31) == 0) red[t >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const int k = fp8_scale_exp(amax);
    const float inv = pow2f(-k);
#pragma unroll
    for (int e = 0; e < 64; e += 2) {
        const uint16_t q = f32x2_to_e4m3x2(v[e + 1] * inv, v[e] * inv);
        tile[cl0 + e][rl] = static_cast<uint8_t>(q & 0xffu);
        tile[cl0 + e + 1][rl] = static_cast<uint8_t>(q >> 8);
    }
    __syncthreads();
    // out column c = cb * 128 + t / 2, bytes (t & 1) * 64 .. +63 of its tile row
    const int cl = t >> 1, h0 = (t & 1) * 64;
    uint4 *dst = reinterpret_cast<uint4 *>(Wq + (static_cast<size_t>(g) * C + cb * QB + cl) * R +
                                           rb * QB + h0);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = *reinterpret_cast<const uint4 *>(&tile[cl][h0 + 16 * i]);
    if (t == 0) S[(static_cast<size_t>(g) * (R / QB) + rb) * (C / QB) + cb] = k;
}

// Rows of bf16 [rows][n] in vectors of 128 -> E4M3 bytes [rows][n] and the vectors' scales
// 2^k as fp32, transposed: sT[n / 128][ld] (a token tile's scales of one 128-wide block
// are then contiguous).  One warp per vector, 4 elements a lane.
__global__ void __launch_bounds__(256) quant_rows_e4m3_kernel(const uint16_t *__restrict__ in,
                                                              long long n_vec, int nb, long long ld,
                                                              uint8_t *__restrict__ out,
                                                              float *__restrict__ sT)
{
    pdl_wait();
    const long long vec = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (vec >= n_vec) return;
    const int lane = threadIdx.x & 31;
    const size_t off = static_cast<size_t>(vec) * QB + 4 * lane;
    const uint2 u = *reinterpret_cast<const uint2 *>(in + off);
    float v[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
    const int k = fp8_scale_exp(amax);
    const float inv = pow2f(-k);
    const uint32_t q01 = f32x2_to_e4m3x2(v[1] * inv, v[0] * inv);
    const uint32_t q23 = f32x2_to_e4m3x2(v[3] * inv, v[2] * inv);
    *reinterpret_cast<uint32_t *>(out + off) = q01 | (q23 << 16);
    if (lane == 0) {
        const long long row = vec / nb, b = vec - row * nb;
        sT[static_cast<size_t>(b) * ld + row] = pow2f(k);
    }
}

// Quantise-dequantise rows of bf16 in vectors of 128: one warp per vector, 4 elements a lane.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t *__restrict__ in,
                                                         long long n_vec, uint16_t *__restrict__ out)
{
    pdl_wait();
    const long long vec = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (vec >= n_vec) return;
    const int lane = threadIdx.x & 31;
    const size_t off = static_cast<size_t>(vec) * QB + 4 * lane;
    const uint2 u = *reinterpret_cast<const uint2 *>(in + off);
    float v[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
    const int k = fp8_scale_exp(amax);
    const float inv = pow2f(-k), sc = pow2f(k);
    const uint16_t q01 = f32x2_to_e4m3x2(v[1] * inv, v[0] * inv);
    const uint16_t q23 = f32x2_to_e4m3x2(v[3] * inv, v[2] * inv);
    const float2 d01 = e4m3x2_to_f32x2(q01), d23 = e4m3x2_to_f32x2(q23);
    uint2 o;
    o.x = f32x2_to_bf16x2(d01.y * sc, d01.x * sc);
    o.y = f32x2_to_bf16x2(d23.y * sc, d23.x * sc);
    *reinterpret_cast<uint2 *>(out + off) = o;
}

}  // namespace

cudaError_t launch_quant_weight(const void *W, int G, int R, int C, void *Wq, int32_t *S,
                                cudaStream_t s)
{
    if (G <= 0 || R <= 0 || C <= 0 || R % QB || C % QB) return cudaErrorInvalidValue;
    return launch_pdl(quant_weight_kernel, dim3(C / QB, R / QB, G), dim3(256), 0, s, 1,
                      static_cast<const uint16_t *>(W), R, C, static_cast<uint8_t *>(Wq), S);
}

cudaError_t launch_quant_rows_e4m3(const void *in, long long rows, int n, void *out, float *sT,
                                   long long ld_sT, cudaStream_t s)
{
    if (rows < 0 || n <= 0 || n % QB || ld_sT < rows) return cudaErrorInvalidValue;
    const long long n_vec = rows * (n / QB);
    if (n_vec == 0) return cudaSuccess;
    return launch_pdl(quant_rows_e4m3_kernel, dim3(static_cast<unsigned>((n_vec + 7) / 8)), dim3(256),
                      0, s, 1, static_cast<const uint16_t *>(in), n_vec, n / QB, ld_sT,
                      static_cast<uint8_t *>(out), sT);
}

cudaError_t launch_quant_rows(const void *in, long long rows, int n, void *out, cudaStream_t s)
{
    if (rows < 0 || n <= 0 || n % QB) return cudaErrorInvalidValue;
    const long long n_vec = rows * (n / QB);
    if (n_vec == 0) return cudaSuccess;
    return launch_pdl(quant_rows_kernel, dim3(static_cast<unsigned>((n_vec + 7) / 8)), dim3(256), 0, s,
                      1, static_cast<const uint16_t *>(in), n_vec, static_cast<uint16_t *>(out));
}

}  // namespace moe
