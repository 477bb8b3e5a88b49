// Glue of the synthetic layer stream: the steps between the GEMMs when M rows are carried from
// layer to layer (the pages give no layer dataflow; the build's reading is h fp32,
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

// bf16 bits of a double, rounded to nearest even in one step: on the bit pattern for results in
// the normal range (the 52-bit mantissa rounded to 7 bits; a carry moves into the exponent, and
// an exponent beyond 127 gives Inf), by an exact scaling to the subnormal quantum 2^-133 below.
__device__ __forceinline__ uint16_t bf16_bits_rne(double v) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(v));
    const uint16_t sign = static_cast<uint16_t>((b >> 48) & 0x8000u);
    const uint64_t a = b & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return 0x7FC0;  // NaN
    const double av = __longlong_as_double(static_cast<long long>(a));
    if (av < 0x1p-126) return sign | static_cast<uint16_t>(rint(av * 0x1p133));  // 128 = smallest normal
    const uint64_t r = (a + 0x0FFFFFFFFFFFull + ((a >> 45) & 1u)) >> 45;  // exponent field | 7 mantissa bits
    const int e = static_cast<int>(r >> 7) - 1023 + 127;
    if (e >= 255) return sign | 0x7F80;
    return sign | static_cast<uint16_t>((e << 7) | static_cast<int>(r & 0x7Fu));
}

// Row m, columns [1024 c, 1024 c + 1024) per block (c = blockIdx.x, m = blockIdx.y): GB300's fp64
// rate is low and a row is short, so the kernel is latency-bound; each block issues all its loads
// of the row at once (16 bytes per thread and round), sums the row's squares in fp64 itself (each
// square of an fp32 value is exact in fp64; a fixed reduction order, so every block gets the same
// sum and the result is reproducible), takes the fp64 reciprocal of sqrt(mean) once, and rounds
// h * that reciprocal once to bf16 (nearest even) for its 1024 columns, which its threads
// already hold. An all-zero row gives zeros. K % 4 == 0, h 16-byte aligned.
constexpr int kRmsChunk = 4 * kRmsThreads;  // columns per block
constexpr int kRmsRound = 8;                // 16-byte loads in flight per thread
__global__ void __launch_bounds__(kRmsThreads) rms_bf16_kernel(const float *__restrict__ h, int K,
                                                               uint16_t *__restrict__ x) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int m = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int K4 = K >> 2;
    const float4 *h4 = reinterpret_cast<const float4 *>(h + static_cast<size_t>(m) * K);
    double s0 = 0.0, s1 = 0.0;
    float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);  // columns 4 (256 c + tid) .. +3
    for (int base = 0; base < K4; base += kRmsThreads * kRmsRound) {
        float4 v[kRmsRound];
#pragma unroll
        for (int j = 0; j < kRmsRound; ++j) {
            const int i = base + j * kRmsThreads + tid;
            v[j] = (i < K4) ? h4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kRmsRound; ++j) {
            s0 = fma(static_cast<double>(v[j].x), static_cast<double>(v[j].x), s0);
            s1 = fma(static_cast<double>(v[j].y), static_cast<double>(v[j].y), s1);
            s0 = fma(static_cast<double>(v[j].z), static_cast<double>(v[j].z), s0);
            s1 = fma(static_cast<double>(v[j].w), static_cast<double>(v[j].w), s1);
            if (base / kRmsThreads + j == c) mine = v[j];
        }
    }
    double ss = s0 + s1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    __shared__ double part[kRmsThreads / 32];
    __shared__ double inv;
    if ((tid & 31) == 0) part[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int i = 0; i < kRmsThreads / 32; ++i) t += part[i];
        const double r = sqrt(t / static_cast<double>(K));
        inv = (r > 0.0) ? 1.0 / r : 0.0;
    }
    __syncthreads();
    const int col = 4 * (c * kRmsThreads + tid);
    if (col < K) {
        const double q = inv;
        uint2 out;
        out.x = static_cast<uint32_t>(bf16_bits_rne(static_cast<double>(mine.x) * q)) |
                (static_cast<uint32_t>(bf16_bits_rne(static_cast<double>(mine.y) * q)) << 16);
        out.y = static_cast<uint32_t>(bf16_bits_rne(static_cast<double>(mine.z) * q)) |
                (static_cast<uint32_t>(bf16_bits_rne(static_cast<double>(mine.w) * q)) << 16);
        *reinterpret_cast<uint2 *>(x + static_cast<size_t>(m) * K + col) = out;
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
    W12_CUDA(cudaLaunchKernelEx(&cfg, rms_bf16_kernel, h, K, x));
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
