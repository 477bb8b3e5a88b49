// The INT6 Q-pass copy (SpecPilot §5.3 "Generality Through Memory": the INT6 copy added for the
// Q pass; App. C: the Q pass reads the nested 8-bit view or a separate low-precision copy).
//
// A separate copy of a weight matrix at 6 bits per weight, 0.75 bytes against the nested view's
// 1.0: per output row a symmetric fp32 scale (the row's largest magnitude over 31) and codes in
// [-31, 31], stored as u = code + 32 in 6 KB records of two planes (low nibbles, top bit pairs)
// laid out so that a decode thread turns one row's 64 codes into bf16 pairs with three shared-
// memory loads and about five instructions per pair. The Q pass is the W12 GEMM kernel reading
// these records (its INT6 mode): codes become exact bf16 integers in registers, the tensor cores
// accumulate x . c in fp32, and each channel's scale is applied as the accumulators leave
// tensor memory.
#include <cuda_bf16.h>

#include "w12_internal.cuh"

namespace w12 {
namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// One warp per row of the copy (padding rows of the last tile included); each lane builds whole
// 64-code record rows, one k tile at a time. The codes are computed with an fp64 division, as
// the copy's definition states (load time only).
__global__ void __launch_bounds__(256) q6_build_kernel(const uint16_t *__restrict__ w, int N, int K, int k_tiles,
                                                       int rows, uint8_t *__restrict__ codes,
                                                       float *__restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (n >= rows) return;
    const int nt = n / 128, nl = n % 128;
    auto store_row = [&](int kt, const uint4 &l0, const uint4 &l1, const uint4 &t) {
        uint8_t *rec = codes + (static_cast<size_t>(nt) * k_tiles + kt) * kQ6RecordBytes;
        *reinterpret_cast<uint4 *>(rec + 16 * nl) = l0;
        *reinterpret_cast<uint4 *>(rec + 2048 + 16 * nl) = l1;
        *reinterpret_cast<uint4 *>(rec + 4096 + 16 * nl) = t;
    };
    // the row's largest magnitude (bf16 bits order like the magnitudes) and whether it holds Inf
    // or NaN
    uint32_t amax_bits = 0;
    bool nonfinite = false;
    const uint16_t *row = w + static_cast<size_t>(n) * K;
    if (n < N) {
        for (int k = lane; k < K; k += 32) {
            const uint32_t a = row[k] & 0x7FFFu;
            nonfinite |= a >= 0x7F80u;
            amax_bits = max(amax_bits, a);
        }
    }
    amax_bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
    nonfinite = __any_sync(0xFFFFFFFFu, nonfinite);
    if (n >= N || nonfinite || amax_bits == 0) {
        // every code 0: u = 32, low nibbles 0, top bit pairs 10b
        const uint4 z = make_uint4(0, 0, 0, 0), t = make_uint4(0xAAAAAAAAu, 0xAAAAAAAAu, 0xAAAAAAAAu, 0xAAAAAAAAu);
        for (int kt = lane; kt < k_tiles; kt += 32) store_row(kt, z, z, t);
        if (lane == 0) scale[n] = 0.f;
        return;
    }
    const float s = static_cast<float>(static_cast<double>(bf16_bits_to_float(amax_bits)) / 31.0);
    const double sd = s;
    for (int kt = lane; kt < k_tiles; kt += 32) {
        uint32_t lw[8] = {0, 0, 0, 0, 0, 0, 0, 0}, tw[4] = {0, 0, 0, 0};
#pragma unroll
        for (int piece = 0; piece < 8; ++piece) {  // 8 weights (16 bytes) each; K % 8 == 0
            const int k0 = kt * 64 + piece * 8;
            const bool valid = k0 < K;
            const uint4 v = valid ? __ldg(reinterpret_cast<const uint4 *>(row + k0)) : make_uint4(0, 0, 0, 0);
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int kl = piece * 8 + e;
                uint32_t u = 32;  // padding columns hold code 0
                if (valid) {
                    const uint32_t bits = (e & 1) ? (vw[e >> 1] >> 16) : (vw[e >> 1] & 0xFFFFu);
                    double t = rint(static_cast<double>(bf16_bits_to_float(bits)) / sd);  // ties to even
                    t = fmin(31.0, fmax(-31.0, t));
                    u = static_cast<uint32_t>(static_cast<int>(t) + 32);
                }
                const int g = kl >> 4, j = (kl & 15) >> 1, h = kl & 1;
                lw[2 * g + (j >> 2)] |= (u & 15u) << (4 * (j & 3) + 16 * h);
                tw[g] |= (u >> 4) << (2 * j + 16 * h);
            }
        }
        store_row(kt, make_uint4(lw[0], lw[1], lw[2], lw[3]), make_uint4(lw[4], lw[5], lw[6], lw[7]),
                  make_uint4(tw[0], tw[1], tw[2], tw[3]));
    }
    if (lane == 0) scale[n] = s;
}

w12_status check_q6(const w12_q6_copy *c) {
    if (!c || !c->codes || !c->scale) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(c->N, c->K));
    if (c->n_tiles != ceil_div(c->N, kTileN) || c->k_tiles != ceil_div(c->K, kTileK)) return W12_ERR_INVALID_ARG;
    if (!aligned16(c->codes)) return W12_ERR_INVALID_ARG;
    return W12_OK;
}

w12_tensor codes_of(const w12_q6_copy *c) {
    w12_tensor t{};
    t.N = c->N;
    t.K = c->K;
    t.n_tiles = c->n_tiles;
    t.k_tiles = c->k_tiles;
    t.records = c->codes;
    return t;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" w12_status w12_q6_shape(int N, int K, w12_q6_copy *c, size_t *codes_bytes, size_t *scale_bytes) {
    if (!c) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(N, K));
    c->N = N;
    c->K = K;
    c->n_tiles = static_cast<int32_t>(ceil_div(N, kTileN));
    c->k_tiles = static_cast<int32_t>(ceil_div(K, kTileK));
    if (codes_bytes) *codes_bytes = static_cast<size_t>(c->n_tiles) * c->k_tiles * kQ6RecordBytes;
    if (scale_bytes) *scale_bytes = sizeof(float) * static_cast<size_t>(c->n_tiles) * kTileN;
    return W12_OK;
}

extern "C" w12_status w12_q6_build(const uint16_t *w, const w12_q6_copy *c, w12_stream_t stream) {
    W12_TRY(check_q6(c));
    if (!w || !aligned16(w)) return W12_ERR_INVALID_ARG;
    int sms = 0;
    W12_TRY(require_device(&sms));
    const int rows = c->n_tiles * kTileN;
    q6_build_kernel<<<(rows + 7) / 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, c->N, c->K, c->k_tiles, rows, c->codes, c->scale);
    W12_CUDA(cudaGetLastError());
    return W12_OK;
}

extern "C" w12_status w12_q6_workspace_size(const w12_q6_copy *c, int M, int argmax, size_t *bytes) {
    W12_TRY(check_q6(c));
    if (!bytes) return W12_ERR_INVALID_ARG;
    const w12_tensor t = codes_of(c);
    return gemm_q6_workspace(&t, M, argmax != 0, bytes);
}

extern "C" w12_status w12_q6_gemm(const w12_q6_copy *c, const uint16_t *x, int M, void *y, int y_dtype,
                                  unsigned flags, void *workspace, size_t workspace_bytes, w12_stream_t stream) {
    W12_TRY(check_q6(c));
    if (flags & ~static_cast<unsigned>(W12_LAUNCH_OVERLAP)) return W12_ERR_INVALID_ARG;
    const w12_tensor t = codes_of(c);
    return gemm_q6(&t, c->scale, x, M, y, y_dtype, workspace, workspace_bytes, stream, flags);
}

extern "C" w12_status w12_q6_argmax(const w12_q6_copy *c, const uint16_t *x, int M, int32_t *idx, float *val,
                                    float *gap, unsigned flags, void *workspace, size_t workspace_bytes,
                                    w12_stream_t stream) {
    W12_TRY(check_q6(c));
    if (flags & ~static_cast<unsigned>(W12_LAUNCH_OVERLAP)) return W12_ERR_INVALID_ARG;
    const w12_tensor t = codes_of(c);
    return gemm_q6_argmax(&t, c->scale, x, M, idx, val, gap, workspace, workspace_bytes, stream, flags);
}
