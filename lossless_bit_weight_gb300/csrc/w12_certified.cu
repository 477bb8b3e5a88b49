// Certified LM head (SpecPilot §4.1 "Certified LM head"): the head also kept as INT8 codes with
// a bound per row (Cauchy-Schwarz on the quantisation residual). A token whose upper bound lies
// below another token's lower bound cannot win and is dropped; the tokens left are scored again
// from the exact weights of the W12 head, with fp32 accumulation; a row that keeps too many
// falls back to the full W12 argmax. The argmax is that of the whole
// head, under the same near-tie rule as the fused argmax: a rescored logit carries fp32
// summation error, so rows whose top-1/top-2 gap is within that error may rank either way.
//
// One call is five stream-ordered launches:
//   1. the GEMM kernel over the INT8 copy (8 KB records of sign-magnitude codes, decoded exactly
//      to bf16 integers in registers, each output channel scaled by its row scale): yh [M, N];
//   2. q8_bounds_kernel: per row, ||x|| and the runner-up L of the lower bounds yh - ||x|| d_n;
//   3. q8_select_kernel: the survivors, tokens whose upper bound yh + ||x|| d_n reaches L (they
//      include the exact top-1 and top-2: the top-1 is at least the best lower bound, and the
//      top-2 at least the smaller of the two best);
//   4. q8_rescore_kernel: each survivor's fp32 logit over the exact weights, from the bf16 head's
//      row when the caller
//      keeps one (contiguous reads) or else from its W12 records and escapes (a gather of
//      16-byte pieces), and the argmax and top-1/top-2 gap over the survivors;
//   5. the W12 fused argmax, which does nothing unless a row had more survivors than the list
//      holds.
// All bounds are evaluated with directed rounding, and the copy's bound d_n includes the fp32
// evaluation error of yh, so that the exact (real-number) logit lies within yh -+ ||x|| d_n.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kQ8RecordBytes = W12_Q8_RECORD_BYTES;
constexpr int kCap = W12_Q8_MAX_SURVIVORS;
constexpr int kBoundThreads = 512;
constexpr int kRescoreThreads = 256;
constexpr int kRescoreWarps = kRescoreThreads / 32;
constexpr int kRescoreBlocksPerRow = 16;
constexpr int kMaxRescoreK = 48 * 1024;  // x row in shared memory as fp32 (+1/64 padding): 195 KB

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// ------------------------------------------------------------------------------------------
// the INT8 copy: one warp per row (padding rows of the last tile included)
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) q8_build_kernel(const uint16_t *__restrict__ w, int N, int K, int k_tiles,
                                                       int rows, uint8_t *__restrict__ codes, float *__restrict__ scale,
                                                       float *__restrict__ bound) {
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (n >= rows) return;
    const int nt = n / 128, nl = n % 128;
    const int chunks = k_tiles * 4;  // 16 codes each
    auto chunk_ptr = [&](int c) {
        return reinterpret_cast<uint4 *>(codes + (static_cast<size_t>(nt) * k_tiles + c / 4) * kQ8RecordBytes +
                                         2048 * (c % 4) + 16 * nl);
    };
    // the row's largest magnitude (as bf16 bits, which order like the values) and whether it
    // holds Inf or NaN
    uint32_t amax_bits = 0;
    bool nonfinite = false;
    if (n < N) {
        const uint16_t *row = w + static_cast<size_t>(n) * K;
        for (int k = lane; k < K; k += 32) {
            const uint32_t a = row[k] & 0x7FFFu;
            nonfinite |= a >= 0x7F80u;
            amax_bits = max(amax_bits, a);
        }
    }
    amax_bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
    nonfinite = __any_sync(0xFFFFFFFFu, nonfinite);
    if (n >= N || nonfinite || amax_bits == 0) {
        for (int c = lane; c < chunks; c += 32) *chunk_ptr(c) = make_uint4(0, 0, 0, 0);
        if (lane == 0) {
            scale[n] = 0.f;
            bound[n] = (n < N && nonfinite) ? INFINITY : 0.f;
        }
        return;
    }
    const float s = static_cast<float>(static_cast<double>(bf16_bits_to_float(amax_bits)) / 127.0);
    const double sd = s;
    const uint16_t *row = w + static_cast<size_t>(n) * K;
    double e2 = 0.0, q2 = 0.0;
    for (int c = lane; c < chunks; c += 32) {
        const int k0 = (c / 4) * 64 + (c % 4) * 16;
        uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int k = k0 + j;
            if (k >= K) break;
            const double wk = bf16_bits_to_float(row[k]);
            double t = rint(wk / sd);  // to nearest, ties to even
            t = fmin(127.0, fmax(-127.0, t));
            const double e = wk - sd * t;  // exact: both terms are exact in fp64
            e2 += e * e;
            q2 += t * t;
            const uint32_t code = (t < 0.0 ? 0x80u : 0u) | static_cast<uint32_t>(fabs(t));
            packed[j >> 2] |= code << (8 * (j & 3));
        }
        *chunk_ptr(c) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        e2 += __shfl_xor_sync(0xFFFFFFFFu, e2, off);
        q2 += __shfl_xor_sync(0xFFFFFFFFu, q2, off);
    }
    if (lane == 0) {
        // residual norm plus the evaluation margin of scale * (x . q) in fp32: each of the K
        // products is exact; the sums (however the tensor cores order and round them) and the
        // final scaling are charged 2^-21 of sum |x_k q_k| <= ||x|| ||q|| per term; the whole
        // is inflated by 2^-16 and rounded up
        const double margin = sd * sqrt(q2) * (static_cast<double>(K) + 3.0) * 0x1p-21;
        const double d = (sqrt(e2) + margin) * (1.0 + 0x1p-16);
        scale[n] = s;
        bound[n] = __double2float_ru(d);
    }
}

// ------------------------------------------------------------------------------------------
// an upper bound on ||x_m||: every square, sum and the square root round upwards, so the
// result bounds the exact norm whatever the order (a square of a bf16 value is exact in fp32
// unless it falls below the normal range, where the upward rounding keeps the bound)
// ------------------------------------------------------------------------------------------
template <int kBlock>
__device__ float row_norm_up(const uint16_t *__restrict__ xm, int K, float *red) {
    float s = 0.f;
#pragma unroll 4
    for (int c = threadIdx.x; c < K / 8; c += kBlock) {  // 16-byte pieces (K % 8 == 0)
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xm) + c);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(wv[j] << 16), b = __uint_as_float(wv[j] & 0xFFFF0000u);
            s = __fadd_ru(s, __fmul_ru(a, a));
            s = __fadd_ru(s, __fmul_ru(b, b));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = __fadd_ru(s, __shfl_xor_sync(0xFFFFFFFFu, s, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < kBlock / 32; ++i) t = __fadd_ru(t, red[i]);
    __syncthreads();
    return __fsqrt_ru(t);
}

// runner-up of the lower bounds per row: blocks (b, m) reduce a slice of n, the last one of a
// row merges the slices
__global__ void __launch_bounds__(kBoundThreads) q8_bounds_kernel(const float *__restrict__ yh, int N,
                                                                  const uint16_t *__restrict__ x, int K,
                                                                  const float *__restrict__ bound, float *rnorm,
                                                                  float2 *lb_top, uint32_t *row_cnt, float *L) {
    __shared__ float red[kBoundThreads / 32];
    __shared__ float2 wtop[kBoundThreads / 32];
    __shared__ int last;
    const int m = blockIdx.y, nb = gridDim.x, b = blockIdx.x;
    const float r = row_norm_up<kBoundThreads>(x + static_cast<size_t>(m) * K, K, red);
    const int n0 = static_cast<int>(static_cast<int64_t>(N) * b / nb);
    const int n1 = static_cast<int>(static_cast<int64_t>(N) * (b + 1) / nb);
    float l1 = -INFINITY, l2 = -INFINITY;
#pragma unroll 4
    for (int n = n0 + threadIdx.x; n < n1; n += kBoundThreads) {
        const float lb = __fsub_rd(yh[static_cast<size_t>(m) * N + n], __fmul_ru(r, bound[n]));
        if (lb > l1) {
            l2 = l1;
            l1 = lb;
        } else if (lb > l2) {
            l2 = lb;
        }
    }
    auto merge = [](float &a1, float &a2, float b1, float b2) {  // the two largest of four
        if (b1 > a1) {
            a2 = fmaxf(a1, b2);
            a1 = b1;
        } else {
            a2 = fmaxf(a2, b1);
        }
    };
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        merge(l1, l2, __shfl_xor_sync(0xFFFFFFFFu, l1, off), __shfl_xor_sync(0xFFFFFFFFu, l2, off));
    if ((threadIdx.x & 31) == 0) wtop[threadIdx.x >> 5] = make_float2(l1, l2);
    __syncthreads();
    if (threadIdx.x == 0) {
        float a1 = -INFINITY, a2 = -INFINITY;
        for (int i = 0; i < kBoundThreads / 32; ++i) merge(a1, a2, wtop[i].x, wtop[i].y);
        lb_top[static_cast<size_t>(m) * nb + b] = make_float2(a1, a2);
        __threadfence();
        last = atomicAdd(&row_cnt[m], 1u) == static_cast<uint32_t>(nb - 1);
    }
    __syncthreads();
    if (last && threadIdx.x < 32) {
        // the slices' results, loaded by the lanes together (nb <= 64), merged by a shuffle tree
        __threadfence();
        float a1 = -INFINITY, a2 = -INFINITY;
        for (int i = threadIdx.x; i < nb; i += 32) {
            const float2 t = __ldcg(&lb_top[static_cast<size_t>(m) * nb + i]);
            merge(a1, a2, t.x, t.y);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            merge(a1, a2, __shfl_xor_sync(0xFFFFFFFFu, a1, off), __shfl_xor_sync(0xFFFFFFFFu, a2, off));
        if (threadIdx.x == 0) {
            L[m] = a2;
            rnorm[m] = r;
            row_cnt[m] = 0;
        }
    }
}

// survivors: tokens whose upper bound reaches L (in no particular order)
__global__ void __launch_bounds__(kBoundThreads) q8_select_kernel(const float *__restrict__ yh, int N,
                                                                  const float *__restrict__ bound,
                                                                  const float *__restrict__ rnorm,
                                                                  const float *__restrict__ L, uint32_t *surv_cnt,
                                                                  int32_t *surv) {
    const int m = blockIdx.y, nb = gridDim.x, b = blockIdx.x;
    const float r = rnorm[m], lm = L[m];
    const int n0 = static_cast<int>(static_cast<int64_t>(N) * b / nb);
    const int n1 = static_cast<int>(static_cast<int64_t>(N) * (b + 1) / nb);
#pragma unroll 4
    for (int n = n0 + threadIdx.x; n < n1; n += kBoundThreads) {
        const float ub = __fadd_ru(yh[static_cast<size_t>(m) * N + n], __fmul_ru(r, bound[n]));
        if (ub >= lm) {
            const uint32_t pos = atomicAdd(&surv_cnt[m], 1u);
            if (pos < static_cast<uint32_t>(kCap)) surv[static_cast<size_t>(m) * kCap + pos] = n;
        }
    }
}

// ------------------------------------------------------------------------------------------
// fp32 rescoring of the survivors over the exact weights of the W12 head
// ------------------------------------------------------------------------------------------
struct W12View {
    const uint16_t *wrow;  // the bf16 head, row-major [N, K], or null (rescore from the records)
    const uint8_t *records;
    const uint8_t *base_exp;
    const uint32_t *esc_off;
    const uint32_t *esc_k;
    const uint16_t *esc_bits;
    int N, K, k_tiles;
};

// x in shared memory with one padding word after every 64: lane l reading k tile l + 32 i then
// hits bank (65 l + j) % 32, all distinct
__device__ __forceinline__ int xs_index(int k) { return k + (k >> 6); }

// y = x . w_n for one row n of the W12 head, by one warp: lane l takes k tiles l, l + 32, ...,
// decodes its 64 weights of each (view bytes and plane B; in a tile that holds one of the row's
// escapes, the escaped weights are replaced as they are used), and the lanes' sums are added by
// a fixed shuffle tree
__device__ float rescore_logit(const W12View &h, int n, const float *xs, int lane) {
    const int nt = n / 128, nl = n % 128;
    const uint32_t base2 = base2_of(h.base_exp[nt * 128 + nl]);
    const uint32_t e0 = h.esc_off[n], e1 = h.esc_off[n + 1];
    // the row's first escapes in registers (rows hold about one on average); a row with more
    // walks its list in memory in the tiles that need it
    constexpr int kRegEsc = 4;
    int ek[kRegEsc];
#pragma unroll
    for (int i = 0; i < kRegEsc; ++i) ek[i] = (e0 + i < e1) ? static_cast<int>(h.esc_k[e0 + i]) : 0x7FFFFFFF;
    const bool many = e1 - e0 > static_cast<uint32_t>(kRegEsc);
    const uint8_t *row0 = h.records + static_cast<size_t>(nt) * h.k_tiles * 12288 + 16 * nl;
    auto load = [&](int kt, uint4 (&c)[6]) {
        const uint8_t *rec = row0 + static_cast<size_t>(kt) * 12288;
        c[0] = __ldg(reinterpret_cast<const uint4 *>(rec + 0 * 2048));
        c[1] = __ldg(reinterpret_cast<const uint4 *>(rec + 1 * 2048));
        c[2] = __ldg(reinterpret_cast<const uint4 *>(rec + 2 * 2048));
        c[3] = __ldg(reinterpret_cast<const uint4 *>(rec + 3 * 2048));
        c[4] = __ldg(reinterpret_cast<const uint4 *>(rec + 8192));
        c[5] = __ldg(reinterpret_cast<const uint4 *>(rec + 8192 + 2048));
    };
    float acc = 0.f;
    uint4 cur[6], nxt[6];
    if (lane < h.k_tiles) load(lane, cur);
    // the next tile's six loads are in flight while this tile is decoded
    for (int kt = lane; kt < h.k_tiles; kt += 32) {
        if (kt + 32 < h.k_tiles) load(kt + 32, nxt);
        uint32_t wd[32];
        decode_chunk16<false, 0>(cur[0], cur[4], base2, wd);
        decode_chunk16<false, 1>(cur[1], cur[4], base2, wd + 8);
        decode_chunk16<false, 0>(cur[2], cur[5], base2, wd + 16);
        decode_chunk16<false, 1>(cur[3], cur[5], base2, wd + 24);
        const int klo = kt * 64;
        const float *xt = xs + xs_index(klo);
        bool has = many;
#pragma unroll
        for (int i = 0; i < kRegEsc; ++i) has |= ek[i] >= klo && ek[i] < klo + 64;
        if (has) {
            // rare: walk the tile's weights against the row's escape list (sorted by k)
            uint32_t e = e0;
            while (e < e1 && static_cast<int>(h.esc_k[e]) < klo) ++e;
            int ke = (e < e1) ? static_cast<int>(h.esc_k[e]) - klo : 64;
            uint32_t bits = (e < e1) ? h.esc_bits[e] : 0u;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                float wv = __uint_as_float((j & 1) ? (wd[j >> 1] & 0xFFFF0000u) : (wd[j >> 1] << 16));
                if (j == ke) {
                    wv = bf16_bits_to_float(bits);
                    ++e;
                    ke = (e < e1) ? static_cast<int>(h.esc_k[e]) - klo : 64;
                    bits = (e < e1) ? h.esc_bits[e] : 0u;
                }
                acc = fmaf(wv, xt[j], acc);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                acc = fmaf(__uint_as_float(wd[j] << 16), xt[2 * j], acc);
                acc = fmaf(__uint_as_float(wd[j] & 0xFFFF0000u), xt[2 * j + 1], acc);
            }
        }
#pragma unroll
        for (int i = 0; i < 6; ++i) cur[i] = nxt[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    return acc;
}

// y = x . w_n from the bf16 head's row n, by one warp: lane l reads the 16-byte pieces l, l + 32,
// ... of the row (K % 8 == 0), and the lanes' sums are added by a fixed shuffle tree
__device__ float rescore_logit_bf16(const W12View &h, int n, const float *xs, int lane) {
    const uint4 *row = reinterpret_cast<const uint4 *>(h.wrow + static_cast<size_t>(n) * h.K);
    const int pieces = h.K / 8;
    float acc = 0.f;
    // four pieces per lane in flight at a time
    for (int c0 = lane; c0 < pieces; c0 += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = (c0 + 32 * u < pieces) ? __ldg(row + c0 + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + 32 * u;
            if (c >= pieces) break;
            const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = 8 * c + 2 * j;
                acc = fmaf(__uint_as_float(wv[j] << 16), xs[xs_index(k)], acc);
                acc = fmaf(__uint_as_float(wv[j] & 0xFFFF0000u), xs[xs_index(k + 1)], acc);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    return acc;
}

__device__ __forceinline__ bool better_logit(float v, int i, float w, int j) { return v > w || (v == w && i < j); }
__device__ __forceinline__ void top2_add(float &v1, int &i1, float &v2, float ov1, int oi1, float ov2) {
    if (better_logit(ov1, oi1, v1, i1)) {
        v2 = fmaxf(ov2, v1);
        v1 = ov1;
        i1 = oi1;
    } else {
        v2 = fmaxf(v2, ov1);
    }
}

__global__ void __launch_bounds__(kRescoreThreads) q8_rescore_kernel(W12View h, const uint16_t *__restrict__ x,
                                                                     uint32_t *surv_cnt, const int32_t *surv,
                                                                     float4 *res_top, uint32_t *res_cnt, int *overflow,
                                                                     int32_t *idx, float *val, float *gap,
                                                                     int32_t *survivors) {
    extern __shared__ float xs[];  // x row as fp32, padded with zeros to k_tiles * 64
    __shared__ float4 wtop[kRescoreWarps];
    __shared__ int last;
    const int m = blockIdx.y, nrb = gridDim.x, b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kpad = h.k_tiles * 64;
    // 16-byte pieces of the row (K % 8 == 0), several loads in flight per thread
#pragma unroll 4
    for (int c = threadIdx.x; c < kpad / 8; c += kRescoreThreads) {
        const int k0 = 8 * c;
        const uint4 v = (k0 < h.K) ? __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(m) * h.K + k0))
                                   : make_uint4(0, 0, 0, 0);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            xs[xs_index(k0 + 2 * j)] = __uint_as_float(wv[j] << 16);
            xs[xs_index(k0 + 2 * j + 1)] = __uint_as_float(wv[j] & 0xFFFF0000u);
        }
    }
    __syncthreads();
    const uint32_t cnt = surv_cnt[m];
    float v1 = -INFINITY, v2 = -INFINITY;
    int i1 = 0x7FFFFFFF;
    if (cnt <= static_cast<uint32_t>(kCap)) {
        for (uint32_t j = b * kRescoreWarps + warp; j < cnt; j += nrb * kRescoreWarps) {
            const int n = surv[static_cast<size_t>(m) * kCap + j];
            float y = h.wrow ? rescore_logit_bf16(h, n, xs, lane) : rescore_logit(h, n, xs, lane);
            if (isnan(y)) y = -INFINITY;  // a NaN logit never wins (as in the fused argmax)
            top2_add(v1, i1, v2, y, n, -INFINITY);
        }
    } else if (threadIdx.x == 0) {
        *overflow = 1;  // the full argmax produces every row's result
    }
    if (lane == 0) wtop[warp] = make_float4(v1, __int_as_float(i1), v2, 0.f);
    __syncthreads();
    if (threadIdx.x == 0) {
        float a1 = -INFINITY, a2 = -INFINITY;
        int ai = 0x7FFFFFFF;
        for (int i = 0; i < kRescoreWarps; ++i) top2_add(a1, ai, a2, wtop[i].x, __float_as_int(wtop[i].y), wtop[i].z);
        res_top[static_cast<size_t>(m) * nrb + b] = make_float4(a1, __int_as_float(ai), a2, 0.f);
        __threadfence();
        last = atomicAdd(&res_cnt[m], 1u) == static_cast<uint32_t>(nrb - 1);
    }
    __syncthreads();
    float a1 = -INFINITY, a2 = -INFINITY;
    int ai = 0x7FFFFFFF;
    if (last && threadIdx.x < 32) {
        // the blocks' results, loaded by the lanes together, merged by a shuffle tree (the top-2
        // of a set does not depend on the merge order)
        __threadfence();
        for (int i = threadIdx.x; i < nrb; i += 32) {
            const float4 t = __ldcg(&res_top[static_cast<size_t>(m) * nrb + i]);
            top2_add(a1, ai, a2, t.x, __float_as_int(t.y), t.z);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o1 = __shfl_xor_sync(0xFFFFFFFFu, a1, off), o2 = __shfl_xor_sync(0xFFFFFFFFu, a2, off);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, ai, off);
            top2_add(a1, ai, a2, o1, oi, o2);
        }
    }
    if (last && threadIdx.x == 0) {
        if (cnt <= static_cast<uint32_t>(kCap)) {
            idx[m] = ai;
            val[m] = a1;
            gap[m] = a1 - a2;
        }
        if (survivors) survivors[m] = static_cast<int32_t>(cnt);
        surv_cnt[m] = 0;
        res_cnt[m] = 0;
    }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
struct CertLayout {
    size_t q8_ws, full_ws;
    size_t off_q8, off_yh, off_rnorm, off_lbtop, off_rowcnt, off_L, off_scnt, off_surv, off_rtop, off_rcnt, off_flag,
        off_full, bytes;
    int nb;
};

w12_tensor codes_tensor(const w12_q8_head *h) {
    w12_tensor c{};
    c.N = h->N;
    c.K = h->K;
    c.n_tiles = h->n_tiles;
    c.k_tiles = h->k_tiles;
    c.records = h->codes;
    return c;
}

w12_status check_q8(const w12_q8_head *h) {
    if (!h || !h->codes || !h->scale || !h->bound) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(h->N, h->K));
    if (h->n_tiles != (h->N + 127) / 128 || h->k_tiles != (h->K + 63) / 64) return W12_ERR_INVALID_ARG;
    if (!aligned16(h->codes)) return W12_ERR_INVALID_ARG;
    return W12_OK;
}

w12_status cert_plan(const w12_tensor *t, const w12_q8_head *h, int M, CertLayout *L) {
    W12_TRY(check_tensor(t));
    W12_TRY(check_q8(h));
    if (t->N != h->N || t->K != h->K) return W12_ERR_INVALID_ARG;
    if (M < 1 || M > W12_MAX_M) return W12_ERR_UNSUPPORTED_SHAPE;
    if (h->k_tiles * 64 > kMaxRescoreK) return W12_ERR_UNSUPPORTED_SHAPE;
    const w12_tensor c = codes_tensor(h);
    W12_TRY(gemm_q8_workspace(&c, M, &L->q8_ws));
    W12_TRY(w12_workspace_size(t, M, W12_OP_ARGMAX, &L->full_ws));
    L->nb = std::max(1, std::min(64, (h->N + 8191) / 8192));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t MN = static_cast<size_t>(M) * h->N;
    L->off_q8 = take(L->q8_ws);
    L->off_full = take(L->full_ws);
    L->off_rowcnt = take(sizeof(uint32_t) * M);
    L->off_scnt = take(sizeof(uint32_t) * M);
    L->off_rcnt = take(sizeof(uint32_t) * M);
    L->off_flag = take(sizeof(int));
    L->off_yh = take(sizeof(float) * MN);
    L->off_rnorm = take(sizeof(float) * M);
    L->off_lbtop = take(sizeof(float2) * static_cast<size_t>(M) * L->nb);
    L->off_L = take(sizeof(float) * M);
    L->off_surv = take(sizeof(int32_t) * static_cast<size_t>(M) * kCap);
    L->off_rtop = take(sizeof(float4) * static_cast<size_t>(M) * kRescoreBlocksPerRow);
    L->bytes = off;
    return W12_OK;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" w12_status w12_q8_shape(int N, int K, w12_q8_head *h, size_t *codes_bytes, size_t *row_bytes) {
    if (!h) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(N, K));
    h->N = N;
    h->K = K;
    h->n_tiles = (N + 127) / 128;
    h->k_tiles = (K + 63) / 64;
    if (codes_bytes) *codes_bytes = static_cast<size_t>(h->n_tiles) * h->k_tiles * kQ8RecordBytes;
    if (row_bytes) *row_bytes = sizeof(float) * static_cast<size_t>(h->n_tiles) * 128;
    return W12_OK;
}

extern "C" w12_status w12_q8_build(const uint16_t *w, const w12_q8_head *h, w12_stream_t stream) {
    W12_TRY(check_q8(h));
    if (!w) return W12_ERR_INVALID_ARG;
    int sms = 0;
    W12_TRY(require_device(&sms));
    const int rows = h->n_tiles * 128;
    q8_build_kernel<<<(rows + 7) / 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w, h->N, h->K, h->k_tiles, rows, h->codes, h->scale, h->bound);
    W12_CUDA(cudaGetLastError());
    return W12_OK;
}

extern "C" w12_status w12_certified_workspace_size(const w12_tensor *t, const w12_q8_head *h, int M,
                                                   size_t *bytes) {
    if (!bytes) return W12_ERR_INVALID_ARG;
    CertLayout L{};
    W12_TRY(cert_plan(t, h, M, &L));
    *bytes = L.bytes;
    return W12_OK;
}

extern "C" w12_status w12_lmhead_certified(const w12_tensor *t, const w12_q8_head *h, const uint16_t *w_bf16,
                                           const uint16_t *x, int M,
                                           int32_t *idx, float *val, float *gap, int32_t *survivors, void *workspace,
                                           size_t workspace_bytes, w12_stream_t stream) {
    CertLayout L{};
    W12_TRY(cert_plan(t, h, M, &L));
    if (!x || !aligned16(x) || !idx || !val || !gap || !workspace) return W12_ERR_INVALID_ARG;
    if (w_bf16 && (!aligned16(w_bf16) || h->K % 8 != 0)) return W12_ERR_INVALID_ARG;
    if (workspace_bytes < L.bytes) return W12_ERR_WORKSPACE;
    int sms = 0;
    W12_TRY(require_device(&sms));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *yh = reinterpret_cast<float *>(ws + L.off_yh);
    float *rnorm = reinterpret_cast<float *>(ws + L.off_rnorm);
    float2 *lbtop = reinterpret_cast<float2 *>(ws + L.off_lbtop);
    uint32_t *rowcnt = reinterpret_cast<uint32_t *>(ws + L.off_rowcnt);
    float *Lrow = reinterpret_cast<float *>(ws + L.off_L);
    uint32_t *scnt = reinterpret_cast<uint32_t *>(ws + L.off_scnt);
    int32_t *surv = reinterpret_cast<int32_t *>(ws + L.off_surv);
    float4 *rtop = reinterpret_cast<float4 *>(ws + L.off_rtop);
    uint32_t *rcnt = reinterpret_cast<uint32_t *>(ws + L.off_rcnt);
    int *flag = reinterpret_cast<int *>(ws + L.off_flag);

    // 1. approximate logits over the INT8 copy
    const w12_tensor c = codes_tensor(h);
    W12_TRY(gemm_q8(&c, h->scale, x, M, yh, ws + L.off_q8, L.q8_ws, stream));
    // 2-3. the runner-up lower bound per row, then the survivors
    const dim3 bg(static_cast<unsigned>(L.nb), static_cast<unsigned>(M));
    q8_bounds_kernel<<<bg, kBoundThreads, 0, st>>>(yh, h->N, x, h->K, h->bound, rnorm, lbtop, rowcnt, Lrow);
    W12_CUDA(cudaGetLastError());
    q8_select_kernel<<<bg, kBoundThreads, 0, st>>>(yh, h->N, h->bound, rnorm, Lrow, scnt, surv);
    W12_CUDA(cudaGetLastError());
    // 4. fp32 rescoring of the survivors over the exact weights
    W12View v{w_bf16, t->records, t->base_exp, t->esc_off, t->esc_k, t->esc_bits, t->N, t->K, t->k_tiles};
    const size_t xs_bytes = sizeof(float) * static_cast<size_t>(t->k_tiles) * 65;
    static std::atomic<uint64_t> smem_set{0};
    int dev = 0;
    W12_CUDA(cudaGetDevice(&dev));
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!bit || !(smem_set.load(std::memory_order_acquire) & bit)) {
        W12_CUDA(cudaFuncSetAttribute(q8_rescore_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(sizeof(float) * (kMaxRescoreK + kMaxRescoreK / 64))));
        smem_set.fetch_or(bit, std::memory_order_acq_rel);
    }
    q8_rescore_kernel<<<dim3(kRescoreBlocksPerRow, static_cast<unsigned>(M)), kRescoreThreads, xs_bytes, st>>>(
        v, x, scnt, surv, rtop, rcnt, flag, idx, val, gap, survivors);
    W12_CUDA(cudaGetLastError());
    // 5. the full argmax, only if a row overflowed its survivor list
    return lmhead_argmax_if(t, x, M, idx, val, gap, flag, ws + L.off_full, L.full_ws, stream);
}

extern "C" w12_status w12_q8_argmax_workspace_size(const w12_q8_head *h, int M, size_t *bytes) {
    W12_TRY(check_q8(h));
    if (!bytes) return W12_ERR_INVALID_ARG;
    const w12_tensor c = codes_tensor(h);
    return gemm_q8_argmax_workspace(&c, M, bytes);
}

extern "C" w12_status w12_q8_argmax(const w12_q8_head *h, const uint16_t *x, int M, int32_t *idx, float *val,
                                    float *gap, unsigned flags, void *workspace, size_t workspace_bytes,
                                    w12_stream_t stream) {
    W12_TRY(check_q8(h));
    if (flags & ~static_cast<unsigned>(W12_LAUNCH_OVERLAP)) return W12_ERR_INVALID_ARG;
    const w12_tensor c = codes_tensor(h);
    return gemm_q8_argmax(&c, h->scale, x, M, idx, val, gap, workspace, workspace_bytes, stream, flags);
}
