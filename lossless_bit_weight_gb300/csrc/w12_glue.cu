// Glue of the synthetic layer stream: the steps between the GEMMs when M rows are carried from
// layer to layer (the pages give no layer dataflow; the reading taken here is h fp32,
// x = bf16(h / rms(h)), a = bf16(x Wq^T), h += a Wo^T, x2 = bf16(h / rms(h)),
// p = bf16((x2 Wg^T) * (x2 Wu^T)), h += p Wd^T). The residual adds are the GEMM's accumulate
// mode; the row normalisation and the gate-up product are the two kernels here. Both are tiny
// (M rows of a few thousand values) and launch-bound, so each one lets the next kernel on the
// stream start at once (a programmatic dependent launch that waits for this one's completion
// before reading its output) and, when launched with W12_LAUNCH_OVERLAP itself, waits for the
// previous kernel's completion only just before it reads its input.
#include <cuda_bf16.h>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kRmsThreads = 256;
constexpr int kMulThreads = 256;

// Row m, columns [1024 c, 1024 c + 1024) per block (c = blockIdx.x, m = blockIdx.y). GB300's fp64
// unit is slow and a row is short, so the kernel is latency-bound; it keeps fp64 off the long
// dependent paths:
//   1. every thread loads its 16-byte pieces of the whole row at once (the block's own 1024
//      columns among them) and the block takes the largest |h|, 2^e its binade;
//   2. the squares of h * 2^-e (at most 1, so nothing overflows) are summed in fp32 pairs
//      (hi, lo) with error-free transformations (the exact square as p + e from an FMA; two-sum
//      additions), across the block in a fixed order: about 2^-40 relative accuracy;
//   3. the mean's reciprocal square root starts from the fp32 approximation and takes one Newton
//      step in fp32 pairs (about 2^-43), kept as an fp32 pair;
//   4. each of the thread's four columns, scaled by 2^-e (exact), is multiplied by it and rounded
//      once to bf16 (fp32 arithmetic; fp64 only for results near the bottom of the fp32 range).
// The result is the bf16 rounding of h / rms(h) except where that quotient lies within about
// 2^-40 (relative) of a rounding boundary. An all-zero row gives zeros. K % 4 == 0, h finite and
// 16-byte aligned.
constexpr int kRmsChunk = 4 * kRmsThreads;  // columns per block
constexpr int kRmsRound = 8;                // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kRmsThreads) rms_bf16_kernel(const float *__restrict__ h, int K, F2 inv_k,
                                                               uint16_t *__restrict__ x) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int m = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int K4 = K >> 2;
    const float4 *h4 = reinterpret_cast<const float4 *>(h + static_cast<size_t>(m) * K);
    const int nround = (K4 + kRmsThreads * kRmsRound - 1) / (kRmsThreads * kRmsRound);
    __shared__ float wmax[kRmsThreads / 32];
    __shared__ F2 wsum[kRmsThreads / 32];
    __shared__ RmsScale scale;
    float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);  // columns 4 (256 c + tid) .. +3
    // pass 1: the largest |h| of the row (rows longer than one round are read again in pass 2)
    float amax = 0.f;
    for (int r = 0; r < nround; ++r) {
        float4 v[kRmsRound];
        const int base = r * kRmsThreads * kRmsRound;
#pragma unroll
        for (int j = 0; j < kRmsRound; ++j) {
            const int i = base + j * kRmsThreads + tid;
            v[j] = (i < K4) ? h4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kRmsRound; ++j) {
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
            if (base / kRmsThreads + j == c) mine = v[j];
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    if ((tid & 31) == 0) wmax[tid >> 5] = amax;
    __syncthreads();
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < kRmsThreads / 32; ++i) bmax = fmaxf(bmax, wmax[i]);
    const int col = 4 * (c * kRmsThreads + tid);
    uint16_t *xr = x + static_cast<size_t>(m) * K;
    if (bmax == 0.f) {  // an all-zero row (block-uniform)
        if (col < K) *reinterpret_cast<uint2 *>(xr + col) = make_uint2(0u, 0u);
        return;
    }
    const int e = ilogbf(bmax) + 1;  // |h| * 2^-e < 1
    // pass 2: the sum of squares of h * 2^-e in fp32 pairs
    F2 acc = {0.f, 0.f};
    for (int r = 0; r < nround; ++r) {
        float4 v[kRmsRound];
        const int base = r * kRmsThreads * kRmsRound;
#pragma unroll
        for (int j = 0; j < kRmsRound; ++j) {
            const int i = base + j * kRmsThreads + tid;
            v[j] = (i < K4) ? h4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kRmsRound; ++j) {
            const float q[4] = {scale_pow2(v[j].x, -e), scale_pow2(v[j].y, -e), scale_pow2(v[j].z, -e),
                                scale_pow2(v[j].w, -e)};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float p = __fmul_rn(q[t], q[t]);
                acc = f2_add(acc, F2{p, __fmaf_rn(q[t], q[t], -p)});  // q^2 = p + that, exactly
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc = f2_add(acc, F2{__shfl_xor_sync(0xFFFFFFFFu, acc.hi, off), __shfl_xor_sync(0xFFFFFFFFu, acc.lo, off)});
    if ((tid & 31) == 0) wsum[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        F2 t = wsum[0];
        for (int i = 1; i < kRmsThreads / 32; ++i) t = f2_add(t, wsum[i]);
        scale = rms_scale(t, inv_k);
    }
    __syncthreads();
    if (col < K) {
        const float yh = scale.yh, yl = scale.yl;
        uint2 out;
        out.x = static_cast<uint32_t>(bf16_mul_rne(scale_pow2(mine.x, -e), yh, yl)) |
                (static_cast<uint32_t>(bf16_mul_rne(scale_pow2(mine.y, -e), yh, yl)) << 16);
        out.y = static_cast<uint32_t>(bf16_mul_rne(scale_pow2(mine.z, -e), yh, yl)) |
                (static_cast<uint32_t>(bf16_mul_rne(scale_pow2(mine.w, -e), yh, yl)) << 16);
        *reinterpret_cast<uint2 *>(xr + col) = out;
    }
}

// p[m, n] = bf16(g[m, n] * u[m, n]): the fp32 product, rounded to nearest even. Row m =
// blockIdx.y; each thread takes four consecutive columns (16-byte loads when the layout allows).
__global__ void __launch_bounds__(kMulThreads) mul_bf16_kernel(const float *__restrict__ g,
                                                               const float *__restrict__ u, int N, int ld,
                                                               int vec, __nv_bfloat16 *__restrict__ p) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int m = blockIdx.y;
    const int n0 = 4 * (blockIdx.x * kMulThreads + threadIdx.x);
    if (n0 >= N) return;
    const float *gr = g + static_cast<size_t>(m) * ld, *ur = u + static_cast<size_t>(m) * ld;
    __nv_bfloat16 *pr = p + static_cast<size_t>(m) * N;
    if (vec) {  // N % 4 == 0, ld % 4 == 0, g, u 16-byte and p 8-byte aligned
        const float4 a = *reinterpret_cast<const float4 *>(gr + n0), b = *reinterpret_cast<const float4 *>(ur + n0);
        __nv_bfloat162 lo, hi;
        lo.x = __float2bfloat16_rn(__fmul_rn(a.x, b.x));
        lo.y = __float2bfloat16_rn(__fmul_rn(a.y, b.y));
        hi.x = __float2bfloat16_rn(__fmul_rn(a.z, b.z));
        hi.y = __float2bfloat16_rn(__fmul_rn(a.w, b.w));
        uint2 out;
        out.x = *reinterpret_cast<const uint32_t *>(&lo);
        out.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(pr + n0) = out;
        return;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (n0 + j < N) pr[n0 + j] = __float2bfloat16_rn(__fmul_rn(gr[n0 + j], ur[n0 + j]));
}

w12_status launch_cfg(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr, unsigned flags, w12_stream_t stream) {
    if (flags & ~static_cast<unsigned>(W12_LAUNCH_OVERLAP)) return W12_ERR_INVALID_ARG;
    cfg->stream = reinterpret_cast<cudaStream_t>(stream);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg->attrs = attr;
    cfg->numAttrs = (flags & W12_LAUNCH_OVERLAP) ? 1 : 0;
    return W12_OK;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" w12_status w12_rms_bf16(const float *h, int M, int K, uint16_t *x, unsigned flags, w12_stream_t stream) {
    if (!h || !x || M < 1 || M > W12_MAX_M || K < 1) return W12_ERR_INVALID_ARG;
    if (K % 4 != 0) return W12_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(h) || (reinterpret_cast<uintptr_t>(x) & 7u) != 0) return W12_ERR_INVALID_ARG;
    int sms = 0;
    W12_TRY(require_device(&sms));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    W12_TRY(launch_cfg(&cfg, attr, flags, stream));
    cfg.gridDim = dim3(static_cast<unsigned>((K + kRmsChunk - 1) / kRmsChunk), static_cast<unsigned>(M));
    cfg.blockDim = dim3(kRmsThreads);
    W12_CUDA(cudaLaunchKernelEx(&cfg, rms_bf16_kernel, h, K, f2_of(1.0 / static_cast<double>(K)), x));
    return W12_OK;
}

extern "C" w12_status w12_mul_bf16(const float *g, const float *u, int M, int N, int ld, uint16_t *p,
                                   unsigned flags, w12_stream_t stream) {
    if (!g || !u || !p || M < 1 || M > W12_MAX_M || N < 1 || ld < N) return W12_ERR_INVALID_ARG;
    int sms = 0;
    W12_TRY(require_device(&sms));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    W12_TRY(launch_cfg(&cfg, attr, flags, stream));
    cfg.gridDim = dim3(static_cast<unsigned>((N + 4 * kMulThreads - 1) / (4 * kMulThreads)), static_cast<unsigned>(M));
    cfg.blockDim = dim3(kMulThreads);
    const int vec = (N % 4 == 0 && ld % 4 == 0 && aligned16(g) && aligned16(u) &&
                     (reinterpret_cast<uintptr_t>(p) & 7u) == 0) ? 1 : 0;
    W12_CUDA(cudaLaunchKernelEx(&cfg, mul_bf16_kernel, g, u, N, ld, vec, reinterpret_cast<__nv_bfloat16 *>(p)));
    return W12_OK;
}
