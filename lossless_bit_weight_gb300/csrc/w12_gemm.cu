// a3/a4/a5 — the skinny W12 GEMM on 5th-generation tensor cores (tcgen05, sm_103a).
//
// SpecPilot §4.1 and Fig. 5b: the GEMM decodes W12 records in registers so that the memory
// stream hides the decode, and splits the reduction over thread blocks in a fixed order so the
// result is deterministic; §6.3 and App. E: it is bound by weight bytes at 1-32 rows; §4.3: the
// Q pass reads only the nested 8-bit view; §2.1: greedy verification takes the row argmax.
//
// Design on GB300 (one persistent block per SM, 16 warps):
//   warp 0       producer: one 1-D bulk copy per 12 KB record (8 KB for the Q view) and one
//                128B-swizzled TMA box of the activations' k-slice per stage
//   warp 1       allocates tensor memory; one thread issues tcgen05.mma (M=128 weight rows from
//                tensor memory, N = rows of x padded to 16 from shared memory, K=16)
//   warp 2       escape feeder: bulk-copies each record's escape entries next to the record
//   warps 4-7    epilogue: tensor memory -> registers; y, split-K partials or the row argmax
//   warps 8-15   two decode groups on alternate records: each thread owns one weight row, turns
//                its 64 view bytes + 32 plane-B bytes into 32 bf16x2 words, patches escapes and
//                stores them into its tensor-memory lane (the MMA's A operand)
// Work split: the R = n_tiles*k_tiles records are cut into `grid` contiguous, equal ranges
// (stream-K). A tile covered by several blocks is finished by whichever arrives last, summing
// the blocks' fp32 partials in increasing block order: no float atomics, bitwise reproducible.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kThreads = 512;
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEscape = 2;
constexpr int kWarpEpi0 = 4;
constexpr int kWarpDec0 = 8;
constexpr int kDecGroups = 2;
constexpr int kEscCap = 256;       // escape entries staged per record; more -> read from global
constexpr int kASlots = 4;         // tensor-memory A buffers (32 columns each)
constexpr int kACols = 32;
constexpr int kAccCol0 = kASlots * kACols;
constexpr int kMaxStages = 8;
constexpr int kMaxM = 256;
constexpr int kSmemLimit = 232448;       // opt-in maximum per block
constexpr int kSmemFloor = 120 * 1024;   // keeps one block per SM
constexpr int kEpiBar = 1;               // named barrier of the 128 epilogue threads

struct Ctrl {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t afull[kASlots], aempty[kASlots];
    uint64_t accfull[2], accempty[2];
    uint64_t done;
    uint32_t esc_hdr[kMaxStages], esc_src[kMaxStages];
    uint32_t tmem_base;
    int abort;
    int fix;
    int pad_;
    float4 wtop[4][kMaxM];  // per-warp top-2 of the current tile (argmax)
    float4 ctop[kMaxM];     // running top-2 of this block (argmax)
};

struct Params {
    const uint8_t *records;
    const uint8_t *base_exp;
    const uint32_t *rec_esc_off;
    const uint32_t *rec_esc;
    int N, K, M, n_tiles, k_tiles, npad, stages, nacc, ncols, grid;
    int64_t R;
    void *y;
    int y_bf16;
    float *partials;     // [grid][2][M][128]
    uint32_t *tile_cnt;  // [n_tiles]
    float4 *cta_top;     // [grid][M]
    uint32_t *done_cnt;  // [1]
    int32_t *idx;
    float *val;
    float *gap;
    int *err;
};

__device__ __forceinline__ int64_t range_start(int64_t c, int64_t R, int64_t G) { return c * R / G; }
// the block whose range holds record i
__device__ __forceinline__ int64_t owner_of(int64_t i, int64_t R, int64_t G) {
    return ((i + 1) * G + R - 1) / R - 1;
}

// ---- argmax helpers: a top-2 is (v1, i1, v2); order = larger value, then smaller index ----
__device__ __forceinline__ bool better(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}
__device__ __forceinline__ void top2_merge(float &v1, int &i1, float &v2, float ov1, int oi1, float ov2) {
    if (better(ov1, oi1, v1, i1)) {
        v2 = fmaxf(ov2, v1);
        v1 = ov1;
        i1 = oi1;
    } else {
        v2 = fmaxf(v2, ov1);
    }
}
__device__ __forceinline__ void warp_top2(float &v1, int &i1, float &v2) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov1 = __shfl_xor_sync(0xFFFFFFFFu, v1, off);
        const int oi1 = __shfl_xor_sync(0xFFFFFFFFu, i1, off);
        const float ov2 = __shfl_xor_sync(0xFFFFFFFFu, v2, off);
        top2_merge(v1, i1, v2, ov1, oi1, ov2);
    }
}

// overwrite one bf16 half of register word `col` (warp-uniform) in the lanes that own it
__device__ __forceinline__ void patch_word(uint32_t (&w)[32], int col, uint32_t keep, uint32_t val) {
#define W12_PATCH_CASE(i) \
    case i: w[i] = (w[i] & keep) | val; break;
    switch (col) {
        W12_PATCH_CASE(0) W12_PATCH_CASE(1) W12_PATCH_CASE(2) W12_PATCH_CASE(3)
        W12_PATCH_CASE(4) W12_PATCH_CASE(5) W12_PATCH_CASE(6) W12_PATCH_CASE(7)
        W12_PATCH_CASE(8) W12_PATCH_CASE(9) W12_PATCH_CASE(10) W12_PATCH_CASE(11)
        W12_PATCH_CASE(12) W12_PATCH_CASE(13) W12_PATCH_CASE(14) W12_PATCH_CASE(15)
        W12_PATCH_CASE(16) W12_PATCH_CASE(17) W12_PATCH_CASE(18) W12_PATCH_CASE(19)
        W12_PATCH_CASE(20) W12_PATCH_CASE(21) W12_PATCH_CASE(22) W12_PATCH_CASE(23)
        W12_PATCH_CASE(24) W12_PATCH_CASE(25) W12_PATCH_CASE(26) W12_PATCH_CASE(27)
        W12_PATCH_CASE(28) W12_PATCH_CASE(29) W12_PATCH_CASE(30) W12_PATCH_CASE(31)
        default: break;
    }
#undef W12_PATCH_CASE
}

template <bool kQView, bool kArgmax>
__global__ void __launch_bounds__(kThreads, 1)
w12_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int S = p.stages;
    const int xbytes = p.npad * 128;
    constexpr int rbytes = kQView ? kViewBytes : kRecordBytes;
    constexpr int ebytes = kQView ? 0 : kEscCap * 4;
    const int sbytes = xbytes + rbytes + ebytes;
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + S * sbytes);
    auto stage_x = [&](int s) { return smem + s * sbytes; };
    auto stage_rec = [&](int s) { return smem + s * sbytes + xbytes; };
    auto stage_esc = [&](int s) { return smem + s * sbytes + xbytes + rbytes; };

    const int c = blockIdx.x;
    const int64_t R = p.R, G = p.grid;
    const int64_t r0 = range_start(c, R, G), r1 = range_start(c + 1, R, G);
    const int nrec = static_cast<int>(r1 - r0);
    const int64_t kt64 = p.k_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&ctrl->full[s]), kQView ? 1 : 2);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int t = 0; t < kASlots; ++t) {
            mbar_init(smem_u32(&ctrl->afull[t]), 128);
            mbar_init(smem_u32(&ctrl->aempty[t]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctrl->accfull[b]), 1);
            mbar_init(smem_u32(&ctrl->accempty[b]), 128);
        }
        mbar_init(smem_u32(&ctrl->done), 1);
        ctrl->abort = 0;
        ctrl->fix = 0;
        fence_barrier_init();
    }
    if (kArgmax) {
        for (int m = threadIdx.x; m < p.M; m += kThreads)
            ctrl->ctop[m] = make_float4(-INFINITY, __int_as_float(0x7FFFFFFF), -INFINITY, 0.f);
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), p.ncols);
        tc_fence_before();
    }
    if (warp == kWarpProducer && lane == 0) prefetch_tensormap(&xmap);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort = &ctrl->abort;
    int issued = 0;  // producer: stages handed to the copy engine; mma: records issued

    if (warp == kWarpProducer) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            for (int j = 0; j < nrec; ++j) {
                const int s = j % S;
                const uint32_t ph = (j / S) & 1;
                if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, abort, p.err, kErrProducer)) break;
                const int64_t r = r0 + j;
                const int kt = static_cast<int>(r % kt64);
                const uint32_t fb = smem_u32(&ctrl->full[s]);
                mbar_arrive_expect_tx(fb, rbytes + xbytes);
                bulk_g2s(smem_u32(stage_rec(s)), p.records + r * kRecordBytes, rbytes, fb);
                tma_2d_g2s(smem_u32(stage_x(s)), &xmap, kt * kTileK, 0, fb);
                issued = j + 1;
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, p.npad);
            int jseg = 0;
            int64_t r = r0;
            bool ok = true;
            while (ok && r < r1) {
                const int64_t tile = r / kt64;
                const int64_t seg_start = r, seg_end = min(r1, (tile + 1) * kt64);
                const int b = (p.nacc == 2) ? (jseg & 1) : 0;
                const uint32_t phb = (p.nacc == 2) ? ((jseg >> 1) & 1) : (jseg & 1);
                if (!mbar_wait(smem_u32(&ctrl->accempty[b]), phb ^ 1, abort, p.err, kErrMma)) break;
                tc_fence_after();
                const uint32_t d = tmem + kAccCol0 + b * p.npad;
                for (; r < seg_end; ++r) {
                    const int j = static_cast<int>(r - r0);
                    const int s = j % S, t = j % kASlots;
                    if (!mbar_wait(smem_u32(&ctrl->full[s]), (j / S) & 1, abort, p.err, kErrMma) ||
                        !mbar_wait(smem_u32(&ctrl->afull[t]), (j / kASlots) & 1, abort, p.err, kErrMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(stage_x(s)));
#pragma unroll
                    for (int kk = 0; kk < kTileK / 16; ++kk)
                        mma_bf16_ts(d, tmem + t * kACols + kk * 8, bdesc + 2 * kk, idesc,
                                    (r != seg_start || kk != 0) ? 1u : 0u);
                    mma_commit(smem_u32(&ctrl->aempty[t]));
                    mma_commit(smem_u32(&ctrl->empty[s]));
                    issued = j + 1;
                }
                if (!ok) break;
                mma_commit(smem_u32(&ctrl->accfull[b]));
                ++jseg;
            }
        }
    } else if (warp == kWarpEscape) {
        // ---------------------------------------------------------------- escape feeder
        if (!kQView) {
            auto load_pair = [&](int base, uint32_t &lo, uint32_t &hi) {
                const int64_t i = r0 + base + lane;
                lo = (i <= R) ? __ldg(p.rec_esc_off + i) : 0u;
                hi = (i + 1 <= R) ? __ldg(p.rec_esc_off + i + 1) : 0u;
            };
            uint32_t lo_c, hi_c, lo_n, hi_n;
            load_pair(0, lo_c, hi_c);
            load_pair(32, lo_n, hi_n);
            for (int j = 0; j < nrec; ++j) {
                if (j > 0 && (j & 31) == 0) {
                    lo_c = lo_n;
                    hi_c = hi_n;
                    load_pair(j + 32, lo_n, hi_n);
                }
                const uint32_t lo = __shfl_sync(0xFFFFFFFFu, lo_c, j & 31);
                const uint32_t hi = __shfl_sync(0xFFFFFFFFu, hi_c, j & 31);
                int ok = 1;
                if (lane == 0) {
                    const int s = j % S;
                    ok = mbar_wait(smem_u32(&ctrl->empty[s]), ((j / S) & 1) ^ 1, abort, p.err, kErrEscape);
                    if (ok) {
                        const uint32_t fb = smem_u32(&ctrl->full[s]);
                        const uint32_t cnt = hi - lo;
                        if (cnt == 0) {
                            ctrl->esc_hdr[s] = 0;
                            mbar_arrive(fb);
                        } else if (cnt <= static_cast<uint32_t>(kEscCap)) {
                            ctrl->esc_hdr[s] = cnt;
                            mbar_arrive_expect_tx(fb, cnt * 4);
                            bulk_g2s(smem_u32(stage_esc(s)), p.rec_esc + lo, cnt * 4, fb);
                        } else {
                            ctrl->esc_hdr[s] = cnt | 0x80000000u;
                            ctrl->esc_src[s] = lo;
                            mbar_arrive(fb);
                        }
                    }
                }
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            }
        }
    } else if (warp >= kWarpDec0) {
        // ---------------------------------------------------------------- decode groups
        const int g = (warp - kWarpDec0) >> 2;
        const int qw = warp & 3;
        const int nl = 32 * qw + lane;
        int64_t cur_tile = -1;
        uint32_t base2 = 0;
        for (int j = g; j < nrec; j += kDecGroups) {
            const int s = j % S, t = j % kASlots;
            const bool ok_full = mbar_wait(smem_u32(&ctrl->full[s]), (j / S) & 1, abort, p.err, kErrDecode);
            if (!__all_sync(0xFFFFFFFFu, ok_full)) break;
            const int64_t r = r0 + j;
            const int64_t tile = r / kt64;
            if (tile != cur_tile) {
                cur_tile = tile;
                base2 = base2_of(__ldg(p.base_exp + tile * kTileN + nl));
            }
            const uint8_t *rec = stage_rec(s);
            uint32_t w[32];
            const uint4 v0 = lds128(rec + 0 * 2048 + 16 * nl);
            const uint4 v1 = lds128(rec + 1 * 2048 + 16 * nl);
            const uint4 v2 = lds128(rec + 2 * 2048 + 16 * nl);
            const uint4 v3 = lds128(rec + 3 * 2048 + 16 * nl);
            if (kQView) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                decode_chunk16<true, 0>(v0, z, base2, w);
                decode_chunk16<true, 1>(v1, z, base2, w + 8);
                decode_chunk16<true, 0>(v2, z, base2, w + 16);
                decode_chunk16<true, 1>(v3, z, base2, w + 24);
            } else {
                const uint4 b0 = lds128(rec + kViewBytes + 16 * nl);
                const uint4 b1 = lds128(rec + kViewBytes + 2048 + 16 * nl);
                decode_chunk16<false, 0>(v0, b0, base2, w);
                decode_chunk16<false, 1>(v1, b0, base2, w + 8);
                decode_chunk16<false, 0>(v2, b1, base2, w + 16);
                decode_chunk16<false, 1>(v3, b1, base2, w + 24);
                // escapes of this record that fall in this warp's 32 rows
                const uint32_t hdr = ctrl->esc_hdr[s];
                const uint32_t cnt = hdr & 0x7FFFFFFFu;
                const bool from_global = (hdr >> 31) != 0;
                const uint32_t *gsrc = p.rec_esc + (from_global ? ctrl->esc_src[s] : 0u);
                const uint32_t *ssrc = reinterpret_cast<const uint32_t *>(stage_esc(s));
                for (uint32_t base = 0; base < cnt; base += 32) {
                    uint32_t e = 0xFFFFFFFFu;
                    if (base + lane < cnt) e = from_global ? __ldg(gsrc + base + lane) : ssrc[base + lane];
                    const uint32_t pos = e & 0xFFFFu;
                    uint32_t mine = __ballot_sync(0xFFFFFFFFu, pos < static_cast<uint32_t>(kRecordWeights) &&
                                                                   (pos >> 11) == static_cast<uint32_t>(qw));
                    while (mine) {
                        const int sl = __ffs(mine) - 1;
                        mine &= mine - 1;
                        const uint32_t ent = __shfl_sync(0xFFFFFFFFu, e, sl);
                        const uint32_t ps = ent & 0xFFFFu;
                        const int owner = static_cast<int>((ps >> 6) & 31u);
                        const int kl = static_cast<int>(ps & 63u);
                        const bool hi = kl & 1;
                        const bool me = lane == owner;
                        const uint32_t keep = me ? (hi ? 0x0000FFFFu : 0xFFFF0000u) : 0xFFFFFFFFu;
                        const uint32_t val = me ? (hi ? (ent & 0xFFFF0000u) : (ent >> 16)) : 0u;
                        patch_word(w, kl >> 1, keep, val);
                    }
                }
            }
            const bool ok_a = mbar_wait(smem_u32(&ctrl->aempty[t]), ((j / kASlots) & 1) ^ 1, abort, p.err, kErrDecode);
            if (!__all_sync(0xFFFFFFFFu, ok_a)) break;
            tc_fence_after();
            tmem_st_32x32b_x32(tmem + (static_cast<uint32_t>(32 * qw) << 16) + t * kACols, w);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&ctrl->afull[t]));
        }
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
        // ---------------------------------------------------------------- epilogue
        const int qw = warp & 3;
        const int nl = 32 * qw + lane;
        const int et = threadIdx.x - kWarpEpi0 * 32;  // 0..127
        const int M = p.M;
        bool dead = false;
        int jseg = 0;
        int64_t r = r0;
        while (r < r1) {
            const int64_t tile = r / kt64;
            const int64_t seg_start = r, seg_end = min(r1, (tile + 1) * kt64);
            r = seg_end;
            const bool full = seg_start == tile * kt64 && seg_end == (tile + 1) * kt64;
            const int slot = (jseg == 0) ? 0 : 1;
            const int b = (p.nacc == 2) ? (jseg & 1) : 0;
            const uint32_t phb = (p.nacc == 2) ? ((jseg >> 1) & 1) : (jseg & 1);
            ++jseg;
            const int n = static_cast<int>(tile) * kTileN + nl;
            bool ok = !dead && mbar_wait(smem_u32(&ctrl->accfull[b]), phb, abort, p.err, kErrEpilogue);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) dead = true;
            float *part = p.partials + (static_cast<size_t>(c) * 2 + slot) * M * kTileN;
            if (!dead) {
                tc_fence_after();
                const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * qw) << 16) + kAccCol0 + b * p.npad;
                for (int m0 = 0; m0 < M; m0 += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tbase + m0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = m0 + i;
                        if (m >= M) break;
                        const float f = __uint_as_float(v[i]);
                        if (!full) {
                            part[static_cast<size_t>(m) * kTileN + nl] = f;
                        } else if (kArgmax) {
                            float v1 = (n < p.N && !isnan(f)) ? f : -INFINITY, v2 = -INFINITY;
                            int i1 = n;
                            warp_top2(v1, i1, v2);
                            if (lane == 0) ctrl->wtop[qw][m] = make_float4(v1, __int_as_float(i1), v2, 0.f);
                        } else if (n < p.N) {
                            if (p.y_bf16)
                                reinterpret_cast<__nv_bfloat16 *>(p.y)[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(f);
                            else
                                reinterpret_cast<float *>(p.y)[static_cast<size_t>(m) * p.N + n] = f;
                        }
                    }
                }
                tc_fence_before();
            }
            mbar_arrive(smem_u32(&ctrl->accempty[b]));

            bool emitted = full;
            if (!full) {
                // split tile: the last block to arrive sums every block's partial in block order
                __threadfence();
                named_bar_sync(kEpiBar, 128);
                if (et == 0) {
                    const int64_t c_lo = owner_of(tile * kt64, R, G);
                    const int64_t c_hi = owner_of((tile + 1) * kt64 - 1, R, G);
                    const uint32_t old = atomicAdd(&p.tile_cnt[tile], 1u);
                    ctrl->fix = (old == static_cast<uint32_t>(c_hi - c_lo)) ? 1 : 0;
                }
                named_bar_sync(kEpiBar, 128);
                emitted = ctrl->fix != 0;
                if (emitted) {
                    __threadfence();
                    const int64_t c_lo = owner_of(tile * kt64, R, G);
                    const int64_t c_hi = owner_of((tile + 1) * kt64 - 1, R, G);
                    for (int m = 0; m < M; ++m) {
                        float f = 0.f;
                        for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
                            const int sl = (range_start(cc, R, G) / kt64 == tile) ? 0 : 1;
                            f += __ldcg(p.partials + ((static_cast<size_t>(cc) * 2 + sl) * M + m) * kTileN + nl);
                        }
                        if (kArgmax) {
                            float v1 = (n < p.N && !isnan(f)) ? f : -INFINITY, v2 = -INFINITY;
                            int i1 = n;
                            warp_top2(v1, i1, v2);
                            if (lane == 0) ctrl->wtop[qw][m] = make_float4(v1, __int_as_float(i1), v2, 0.f);
                        } else if (n < p.N) {
                            if (p.y_bf16)
                                reinterpret_cast<__nv_bfloat16 *>(p.y)[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(f);
                            else
                                reinterpret_cast<float *>(p.y)[static_cast<size_t>(m) * p.N + n] = f;
                        }
                    }
                    if (et == 0) p.tile_cnt[tile] = 0;  // leave the workspace zeroed
                }
            }
            if (kArgmax && emitted) {
                named_bar_sync(kEpiBar, 128);
                for (int m = et; m < M; m += 128) {
                    float4 a = ctrl->ctop[m];
                    float v1 = a.x, v2 = a.z;
                    int i1 = __float_as_int(a.y);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 o = ctrl->wtop[q][m];
                        top2_merge(v1, i1, v2, o.x, __float_as_int(o.y), o.z);
                    }
                    ctrl->ctop[m] = make_float4(v1, __int_as_float(i1), v2, 0.f);
                }
                named_bar_sync(kEpiBar, 128);
            }
        }
        if (kArgmax) {
            // publish this block's top-2 per row; the last block merges all blocks in order
            for (int m = et; m < M; m += 128) p.cta_top[static_cast<size_t>(c) * M + m] = ctrl->ctop[m];
            __threadfence();
            named_bar_sync(kEpiBar, 128);
            if (et == 0) {
                const uint32_t old = atomicAdd(p.done_cnt, 1u);
                ctrl->fix = (old == static_cast<uint32_t>(G - 1)) ? 1 : 0;
            }
            named_bar_sync(kEpiBar, 128);
            if (ctrl->fix) {
                __threadfence();
                for (int m = et; m < M; m += 128) {
                    float v1 = -INFINITY, v2 = -INFINITY;
                    int i1 = 0x7FFFFFFF;
                    for (int64_t cc = 0; cc < G; ++cc) {
                        const float4 o = __ldcg(p.cta_top + static_cast<size_t>(cc) * M + m);
                        top2_merge(v1, i1, v2, o.x, __float_as_int(o.y), o.z);
                    }
                    p.idx[m] = i1;
                    p.val[m] = v1;
                    p.gap[m] = v1 - v2;
                }
                if (et == 0) *p.done_cnt = 0;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (warp == kWarpProducer && lane == 0 && ctrl->abort) {
        // let copies still in flight land before the block's shared memory is released
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
            if (!mbar_wait_drain(smem_u32(&ctrl->full[j % S]), (j / S) & 1)) atomicOr(p.err, kErrDrain);
    }
    if (warp == kWarpMma) {
        if (lane == 0 && issued > 0) {
            mma_commit(smem_u32(&ctrl->done));
            if (!mbar_wait_drain(smem_u32(&ctrl->done), 0)) atomicOr(p.err, kErrDrain);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, p.ncols);
    }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

struct Layout {
    int npad, stages, nacc, ncols, grid, smem;
    int64_t R;
    size_t ws_bytes, off_err, off_tile, off_done, off_part, off_top;
};

w12_status plan(const w12_tensor *t, int M, int op, Layout *L) {
    if (M < 1 || M > kMaxM) return W12_ERR_UNSUPPORTED_SHAPE;
    if (op < W12_OP_GEMM || op > W12_OP_QVIEW_ARGMAX) return W12_ERR_INVALID_ARG;
    int sms = 0;
    W12_TRY(require_device(&sms));
    const bool q = (op == W12_OP_QVIEW_GEMM || op == W12_OP_QVIEW_ARGMAX);
    L->R = static_cast<int64_t>(t->n_tiles) * t->k_tiles;
    L->npad = (M + 15) / 16 * 16;
    const int sbytes = L->npad * 128 + (q ? kViewBytes : kRecordBytes) + (q ? 0 : kEscCap * 4);
    const int ctrl = static_cast<int>(align_up(sizeof(Ctrl), 1024));
    L->stages = (kSmemLimit - 1024 - ctrl) / sbytes;
    if (L->stages > kMaxStages) L->stages = kMaxStages;
    if (L->stages < 2) return W12_ERR_UNSUPPORTED_SHAPE;
    L->smem = 1024 + L->stages * sbytes + ctrl;
    if (L->smem < kSmemFloor) L->smem = kSmemFloor;
    L->nacc = (kAccCol0 + 2 * L->npad <= 512) ? 2 : 1;
    const int cols = kAccCol0 + L->nacc * L->npad;
    L->ncols = cols <= 256 ? 256 : 512;
    L->grid = static_cast<int>(L->R < sms ? L->R : sms);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L->off_err = take(16);
    L->off_tile = take(sizeof(uint32_t) * t->n_tiles);
    L->off_done = take(16);
    L->off_part = take(sizeof(float) * static_cast<size_t>(L->grid) * 2 * M * kTileN);
    L->off_top = take(sizeof(float4) * static_cast<size_t>(L->grid) * M);
    L->ws_bytes = off;
    return W12_OK;
}

template <bool kQ, bool kA>
w12_status launch_variant(const CUtensorMap &map, const Params &p, const Layout &L, cudaStream_t st) {
    auto kern = w12_gemm_kernel<kQ, kA>;
    W12_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem));
    kern<<<L.grid, kThreads, L.smem, st>>>(map, p);
    W12_CUDA(cudaGetLastError());
    return W12_OK;
}

w12_status run(const w12_tensor *t, const uint16_t *x, int M, int op, void *y, int y_dtype,
               int32_t *idx, float *val, float *gap, void *ws, size_t ws_bytes, w12_stream_t stream) {
    W12_TRY(check_tensor(t));
    if (!x || !aligned16(x) || !ws) return W12_ERR_INVALID_ARG;
    Layout L{};
    W12_TRY(plan(t, M, op, &L));
    if (ws_bytes < L.ws_bytes) return W12_ERR_WORKSPACE;
    const bool argmax = (op == W12_OP_ARGMAX || op == W12_OP_QVIEW_ARGMAX);
    const bool q = (op == W12_OP_QVIEW_GEMM || op == W12_OP_QVIEW_ARGMAX);
    if (argmax && (!idx || !val || !gap)) return W12_ERR_INVALID_ARG;
    if (!argmax && (!y || (y_dtype != W12_OUT_F32 && y_dtype != W12_OUT_BF16))) return W12_ERR_INVALID_ARG;

    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return W12_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(t->K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(t->K) * 2};
    const cuuint32_t box[2] = {kTileK, static_cast<cuuint32_t>(L.npad)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return W12_ERR_INVALID_ARG;

    uint8_t *w = static_cast<uint8_t *>(ws);
    Params p{};
    p.records = t->records;
    p.base_exp = t->base_exp;
    p.rec_esc_off = t->rec_esc_off;
    p.rec_esc = t->rec_esc;
    p.N = t->N;
    p.K = t->K;
    p.M = M;
    p.n_tiles = t->n_tiles;
    p.k_tiles = t->k_tiles;
    p.npad = L.npad;
    p.stages = L.stages;
    p.nacc = L.nacc;
    p.ncols = L.ncols;
    p.grid = L.grid;
    p.R = L.R;
    p.y = y;
    p.y_bf16 = (y_dtype == W12_OUT_BF16);
    p.err = reinterpret_cast<int *>(w + L.off_err);
    p.tile_cnt = reinterpret_cast<uint32_t *>(w + L.off_tile);
    p.done_cnt = reinterpret_cast<uint32_t *>(w + L.off_done);
    p.partials = reinterpret_cast<float *>(w + L.off_part);
    p.cta_top = reinterpret_cast<float4 *>(w + L.off_top);
    p.idx = idx;
    p.val = val;
    p.gap = gap;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (q) return argmax ? launch_variant<true, true>(map, p, L, st) : launch_variant<true, false>(map, p, L, st);
    return argmax ? launch_variant<false, true>(map, p, L, st) : launch_variant<false, false>(map, p, L, st);
}

}  // namespace
}  // namespace w12

extern "C" w12_status w12_workspace_size(const w12_tensor *t, int M, int op, size_t *bytes) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    if (!bytes) return W12_ERR_INVALID_ARG;
    Layout L{};
    W12_TRY(plan(t, M, op, &L));
    *bytes = L.ws_bytes;
    return W12_OK;
}

extern "C" w12_status w12_gemm_config(const w12_tensor *t, int M, int op, int *grid, int *stages,
                                      int *smem_bytes) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    Layout L{};
    W12_TRY(plan(t, M, op, &L));
    if (grid) *grid = L.grid;
    if (stages) *stages = L.stages;
    if (smem_bytes) *smem_bytes = L.smem;
    return W12_OK;
}

extern "C" w12_status w12_gemm(const w12_tensor *t, const uint16_t *x, int M, void *y, int y_dtype,
                               void *workspace, size_t workspace_bytes, w12_stream_t stream) {
    return w12::run(t, x, M, W12_OP_GEMM, y, y_dtype, nullptr, nullptr, nullptr, workspace,
                    workspace_bytes, stream);
}

extern "C" w12_status w12_qview_gemm(const w12_tensor *t, const uint16_t *x, int M, void *y,
                                     int y_dtype, void *workspace, size_t workspace_bytes,
                                     w12_stream_t stream) {
    return w12::run(t, x, M, W12_OP_QVIEW_GEMM, y, y_dtype, nullptr, nullptr, nullptr, workspace,
                    workspace_bytes, stream);
}

extern "C" w12_status w12_lmhead_argmax(const w12_tensor *t, const uint16_t *x, int M, int32_t *idx,
                                        float *val, float *gap, int qview, void *workspace,
                                        size_t workspace_bytes, w12_stream_t stream) {
    return w12::run(t, x, M, qview ? W12_OP_QVIEW_ARGMAX : W12_OP_ARGMAX, nullptr, W12_OUT_F32, idx,
                    val, gap, workspace, workspace_bytes, stream);
}

extern "C" w12_status w12_check(void *workspace, size_t workspace_bytes, w12_stream_t stream) {
    if (!workspace || workspace_bytes < 16) return W12_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int err = 0;
    if (cudaMemcpyAsync(&err, workspace, sizeof err, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return W12_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return W12_ERR_CUDA;
    if (err) {
        if (cudaMemsetAsync(workspace, 0, sizeof err, st) != cudaSuccess) return W12_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return W12_ERR_CUDA;
        return W12_ERR_TIMEOUT;
    }
    return W12_OK;
}
