// f3 — the persistent cross-GEMM W12 kernel (SpecPilot App. F and Table A7: one kernel that
// runs a sequence of W12 GEMMs instead of a launch per GEMM; the pages measured it on H100 and
// closed it there).
//
// One cooperative launch runs a whole decoding step of the synthetic layer stream (the pages give
// no layer dataflow; the reading taken here carries M rows h fp32 from layer to layer):
//   per layer   x  = bf16(h / rms(h))                       row-normalisation phase
//               qkv = bf16(x Wqkv^T)                        GEMM (k and v are computed and dropped)
//               h += qkv[:, :n_q] Wo^T                      GEMM, added into h
//               x2 = bf16(h / rms(h))                       row-normalisation phase
//               p  = bf16((x2 Wg^T) * (x2 Wu^T))            GEMM, product fused into its epilogue
//               h += p Wd^T                                 GEMM, added into h
//   at the end  x_out = bf16(h / rms(h))                    row-normalisation phase
// The arithmetic is that of the separate calls (w12_gemm with the same work split, w12_rms_bf16,
// w12_mul_bf16, the accumulate mode), so the step gives the same rows as the chain of launches.
//
// Design on GB300: one block per SM (cooperative launch, so all blocks are resident), the warp
// roles of the W12 GEMM kernel (activation producer, two MMA issuers, a feeder of records and
// escape words, four epilogue warps, three decode groups of four warps) and a sequence of slots
// (two records each) that runs through every GEMM of the step. Weights are static, so the feeder
// keeps fetching the records of the next GEMM into free shared-memory slots and the decode groups
// keep decoding them into free tensor-memory slots while the previous phase is still finishing;
// only the activation copies of a GEMM wait, until every block has completed the phase that
// writes them (a per-phase completion counter in global memory, polled with a bounded wait). The
// two kinds of slot form rings of their own, so at a phase boundary both shared and tensor memory
// hold the next phase's weights. The epilogue warps write each GEMM's outputs (a tile split
// between blocks is summed in increasing block order, each of the tile's blocks summing a slice of
// it; gate|up's by the block that publishes its part last) and run the row-normalisation phases. The gate and up rows are interleaved in blocks of 64 at load time, so
// a 128-row tile holds 64 gate rows and the 64 matching up rows and its epilogue forms the
// product. Every wait is bounded (about a second); a block that gives up records an error bit in
// the workspace error word and stops.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <new>

#include "w12_internal.cuh"

namespace w12 {

namespace {

constexpr int kDecGroupsS = 3;
constexpr int kThreadsS = 32 * (8 + 4 * kDecGroupsS);
constexpr int kWProducer = 0, kWMma = 1, kWEscape = 2, kWMma2 = 3, kWEpi0 = 4, kWDec0 = 8;
constexpr int kEscCapS = 112;      // index words staged per slot; more -> read from global
constexpr int kAColsS = 32;        // tensor-memory columns of one decoded record
constexpr int kMaxStagesS = 8;     // slots of decoded records in tensor memory (and their activations)
constexpr int kMaxRawS = 10;       // slots of copied records in shared memory
constexpr int kRowF4 = 10;  // 16-byte words of a row one epilogue thread holds in a normalisation unit
constexpr int kTmemColsS = 512;
constexpr int kSmemLimitS = 232448;
constexpr int kEpiBarS = 1;
constexpr int kKinds = 4;          // q|k|v, o, gate|up, down
constexpr int kKindQkv = 0, kKindO = 1, kKindGu = 2, kKindDown = 3;
constexpr int kPhasesPerLayer = 6;  // rms, q|k|v, o, rms, gate|up, down
constexpr int kMaxLayersS = W12_STREAM_MAX_LAYERS;
constexpr int kMaxMS = W12_STREAM_MAX_M;
constexpr uint32_t kAllOnes = 0xFFFFFFFFu;

// phase index (within a layer) of each GEMM kind
__device__ __forceinline__ int gemm_phase(int gp) {
    const int k = gp & 3;
    return kPhasesPerLayer * (gp >> 2) + ((k < 2) ? k + 1 : k + 2);
}

struct STensor {  // the device buffers one GEMM reads
    const uint8_t *records;
    const uint8_t *base_exp;
    const uint32_t *rec_esc_off;
    const uint32_t *rec_esc;
};

struct SKind {  // shape and work split of one of the four linears (the same in every layer)
    int N, K, n_tiles, k_tiles, R;
    int unit;   // records per work unit: k_tiles (whole tiles) or 1 (stream-K)
    int grid;   // blocks that share the work (the rest get none)
};

struct SParams {
    STensor t[kMaxLayersS][kKinds];
    SKind kind[kKinds];
    int L, M, npad, stages, rstages, nacc, acc_cols, G, H, F, Nqkv, rms_chunks, sbytes;
    F2 inv_h;  // 1 / H as an fp32 pair
    float *h;
    uint16_t *xa, *xm, *qkv, *pg, *x_out;
    float *partials;     // [2][G][2][M][128]
    uint32_t *tile_cnt;  // [kKinds][max_tiles]
    int max_tiles;
    uint32_t *done;      // [6 L + 1] blocks that completed each phase
    int *err;
    uint32_t m3, m15;
    int test_stall;  // W12_LAUNCH_TEST_STALL: the producer issues its first slot's copies only
};

struct SCtrl {
    uint64_t full[kMaxRawS], rfree[kMaxRawS];                        // copied-record slots
    uint64_t afull[kMaxStagesS], empty[kMaxStagesS], xfull[kMaxStagesS];  // decoded slots
    uint64_t accfull[2], accempty[2];
    uint64_t drained[2];
    uint2 esc_info[kMaxRawS];
    const uint32_t *esc_ptr[kMaxRawS];  // the slot's index words in global memory (when not staged)
    int slot_nr[kMaxRawS];              // records in the slot (1 or 2)
    int slot_en1[kMaxRawS];             // offset of the second record's window bases (0: same tile)
    int nslots;                            // slots in the block's whole sequence
    uint32_t tmem_base;
    int abort;
    int last;            // this block published a split tile's part last and sums it
    float red_max[4];    // the row normalisation's cross-warp reductions
    F2 red_sum[4];
    RmsScale scale;
};
constexpr size_t kSCtrlBytes = (sizeof(SCtrl) + 127) / 128 * 128;
constexpr size_t kXchgBytes = 16 * 64 * 4;  // up-half values of 16 rows x 64 columns
constexpr int kEnBytes = 2 * kTileN;        // a slot's window bases E_n: 128 rows per record
// a copied-record slot: two records, the index words, the window bases
constexpr int kRawBytes = 2 * kRecordBytes + kEscCapS * 4 + kEnBytes;
static_assert(kRawBytes % 16 == 0, "bulk copies land on 16-byte boundaries");

__device__ __forceinline__ int range_start_s(int c, int units, int G) {
    return static_cast<int>(static_cast<uint32_t>(c) * static_cast<uint32_t>(units) / static_cast<uint32_t>(G));
}
__device__ __forceinline__ int owner_of_s(int i, int units, int G) {
    return static_cast<int>((static_cast<uint32_t>(i + 1) * G + units - 1) / static_cast<uint32_t>(units)) - 1;
}

struct RingS {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance(int by, int size) {
        idx += by;
        while (idx >= size) {
            idx -= size;
            phase ^= 1u;
        }
    }
};

// This block's record range [r0, r1) in GEMM phase gp.
__device__ __forceinline__ void block_range(const SParams &p, int gp, int c, int &r0, int &r1) {
    const SKind &k = p.kind[gp & 3];
    if (c >= k.grid) {
        r0 = r1 = 0;
        return;
    }
    const int units = k.R / k.unit;
    r0 = k.unit * range_start_s(c, units, k.grid);
    r1 = k.unit * range_start_s(c + 1, units, k.grid);
}

// Position in the block's sequence of ring slots: GEMM phase gp, the slot's first record r, the
// end of the block's range in that phase, the slot's record count and its global index.
struct SlotIt {
    int gp, r, r1, nr, js;
    __device__ __forceinline__ void seek(const SParams &p, int c) {  // first non-empty phase from gp
        while (gp < 4 * p.L) {
            int a, b;
            block_range(p, gp, c, a, b);
            if (a < b) {
                r = a;
                r1 = b;
                nr = min(2, r1 - r);
                return;
            }
            ++gp;
        }
        r = r1 = nr = 0;
    }
    __device__ __forceinline__ void next(const SParams &p, int c) {
        r += nr;
        ++js;
        if (r >= r1) {
            ++gp;
            seek(p, c);
        } else {
            nr = min(2, r1 - r);
        }
    }
    __device__ __forceinline__ bool end(const SParams &p) const { return gp >= 4 * p.L; }
};

// Bounded wait until *cnt >= target (another phase completed on every block); one thread polls.
__device__ __forceinline__ bool wait_count(const uint32_t *cnt, uint32_t target, volatile int *abort, int *gerr,
                                           int code) {
    if (ld_acquire_gpu(cnt) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(128);
        if (ld_acquire_gpu(cnt) >= target) return true;
        if ((it & 7u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(gerr, code);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The activations of each GEMM kind, as kernel parameters of their own (like the GEMM kernel's):
// one 64-wide k slice (a*) and two consecutive slices in one copy (b*), for q|k|v, o, gate|up
// and down.
__global__ void __launch_bounds__(kThreadsS, 1)
w12_stream_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap b0,
                  const __grid_constant__ CUtensorMap a1, const __grid_constant__ CUtensorMap b1,
                  const __grid_constant__ CUtensorMap a2, const __grid_constant__ CUtensorMap b2,
                  const __grid_constant__ CUtensorMap a3, const __grid_constant__ CUtensorMap b3,
                  const __grid_constant__ SParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_launch_dependents();  // the next kernel may start loading its weights as SMs free up
    // Two rings. Copied records (with their index words and window bases) occupy a shared-memory
    // slot (Sm of them) only until a decode group has moved them into tensor memory; the decoded
    // records and the slot's activations then wait in one of St tensor-memory slots for the MMAs.
    // So while the MMAs wait at a phase boundary, Sm + St slots of the next phase are in flight
    // or ready.
    const int S = p.stages, Sm = p.rstages, M = p.M, G = p.G, L = p.L;
    const int xbytes = p.npad * 128;
    const int sbytes = p.sbytes;  // the two activation tiles of a tensor-memory slot
    uint8_t *raw = smem + S * sbytes;
    SCtrl *ctrl = reinterpret_cast<SCtrl *>(raw + Sm * kRawBytes);
    float *xchg = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ctrl) + kSCtrlBytes);
    auto stage_x = [&](int s, int q) { return smem + s * sbytes + q * xbytes; };
    auto stage_rec = [&](int m, int q) { return raw + m * kRawBytes + q * kRecordBytes; };
    auto stage_esc = [&](int m) { return raw + m * kRawBytes + 2 * kRecordBytes; };
    auto stage_en = [&](int m) { return raw + m * kRawBytes + 2 * kRecordBytes + kEscCapS * 4; };
    const int c = blockIdx.x;
    const uint32_t Gu = static_cast<uint32_t>(G);

    if (warp == kWProducer) {
        if (lane == 0) {
            for (int m = 0; m < Sm; ++m) {
                mbar_init(smem_u32(&ctrl->full[m]), 1);     // the escape feeder's copies
                mbar_init(smem_u32(&ctrl->rfree[m]), 128);  // the decode group is done with them
            }
            for (int s = 0; s < S; ++s) {
                mbar_init(smem_u32(&ctrl->afull[s]), 128);
                mbar_init(smem_u32(&ctrl->empty[s]), 2);  // one arrival per MMA issuer
                mbar_init(smem_u32(&ctrl->xfull[s]), 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&ctrl->accfull[b]), 2);
                mbar_init(smem_u32(&ctrl->accempty[b]), 128);
                mbar_init(smem_u32(&ctrl->drained[b]), 1);
            }
            ctrl->abort = 0;
            int ns = 0;
            for (int gp = 0; gp < 4 * L; ++gp) {
                int a, b;
                block_range(p, gp, c, a, b);
                ns += (b - a + 1) >> 1;
            }
            ctrl->nslots = ns;
            fence_barrier_init();
            prefetch_tensormap(&a0);
            prefetch_tensormap(&b0);
            prefetch_tensormap(&a1);
            prefetch_tensormap(&b1);
            prefetch_tensormap(&a2);
            prefetch_tensormap(&b2);
            prefetch_tensormap(&a3);
            prefetch_tensormap(&b3);
        }
        __syncwarp();
    }
    if (warp == kWMma) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemColsS);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    auto a_slot = [&](int s, int q) { return tmem + p.acc_cols + (s * 2 + q) * kAColsS; };
    volatile int *abort = &ctrl->abort;
    int issued = 0;   // escape feeder: slots whose records were requested
    int xissued = 0;  // producer: slots whose activations were requested
    int mma_issued = 0;           // issuers: slots they issued MMAs for

    SlotIt start;
    start.gp = 0;
    start.js = 0;
    start.seek(p, c);

    if (warp == kWProducer) {
        // ---------------------------------------------------------------- producer (warp-wide)
        // Activation tiles of each slot, in slot order: once the slot's tensor-memory position is
        // free (its tiles sit beside it) and the phase that writes the GEMM's input has completed
        // on every block. The records of the slots go out from the escape feeder, which runs up to
        // both rings' depth ahead of the activations, across GEMM boundaries. This loop stays
        // short: the warp shares its scheduler with three decode warps, and every instruction here
        // delays the next copy.
        SlotIt xi = start;
        RingS xr;
        int known = 0;  // phases [0, known) are known to be complete on every block
        // the current GEMM phase's constants, loaded once per phase (parameter reads with run-time
        // indices are slow)
        int xgp = -1, xKT = 1, xkt = 0, xneed = 0;
        const CUtensorMap *xm1 = nullptr, *xm2 = nullptr;
        while (!xi.end(p)) {
            const bool okf = mbar_wait(smem_u32(&ctrl->empty[xr.idx]), xr.phase ^ 1u, abort, p.err, kErrProducer);
            if (!__all_sync(kAllOnes, okf)) break;
            if (xi.gp != xgp) {
                xgp = xi.gp;
                const int k = xgp & 3;
                xKT = p.kind[k].k_tiles;
                xkt = xi.r % xKT;
                xm1 = (k == 0) ? &a0 : (k == 1) ? &a1 : (k == 2) ? &a2 : &a3;
                xm2 = (k == 0) ? &b0 : (k == 1) ? &b1 : (k == 2) ? &b2 : &b3;
                xneed = gemm_phase(xgp) - 1;  // the phase that writes this GEMM's input
            }
            if (xneed >= known) {
                bool okp = true;
                if (lane == 0) okp = wait_count(p.done + xneed, Gu, abort, p.err, kErrProducer);
                if (!__shfl_sync(kAllOnes, okp, 0)) break;
                known = xneed + 1;
                fence_proxy_async_global();  // generic writes of other SMs before async reads
            }
            const uint32_t xb = smem_u32(&ctrl->xfull[xr.idx]);
            mbar_arrive_expect_tx_elect(xb, static_cast<uint32_t>(xi.nr * xbytes));
            if (xi.nr == 2 && xkt + 1 < xKT) {
                tma_3d_g2s_elect(smem_u32(stage_x(xr.idx, 0)), xm2, 0, 0, xkt, xb);
            } else {
                tma_2d_g2s_elect(smem_u32(stage_x(xr.idx, 0)), xm1, xkt * kTileK, 0, xb);
                if (xi.nr == 2)
                    tma_2d_g2s_elect(smem_u32(stage_x(xr.idx, 1)), xm1, ((xkt + 1) % xKT) * kTileK, 0, xb);
            }
            xkt += xi.nr;
            while (xkt >= xKT) xkt -= xKT;
            xi.next(p, c);
            xr.advance(1, S);
            xissued = xi.js;
            if (p.test_stall) break;  // the test hook: the MMAs' wait on the next slot runs out
        }
    } else if (warp == kWMma || warp == kWMma2) {
        // ---------------------------------------------------------------- MMA issuers (warp-wide)
        // Issuer mq takes record mq of every slot into an accumulator of its own; per segment (the
        // block's part of one tile) it overwrites its accumulator with its first record, adds the
        // rest and commits accfull. A slot with one record gets an arrival on empty from issuer 1
        // once that slot has been refilled (after its afull), so its next use is not released early.
        const int mq = (warp == kWMma) ? 0 : 1;
        const uint32_t idesc = idesc_bf16_f32(128, p.npad);
        const uint64_t bstep = static_cast<uint64_t>(sbytes >> 4);
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(stage_x(0, mq)));
        const uint32_t astep = static_cast<uint32_t>(2 * kAColsS);
        RingS st;
        int js_cur = 0;  // global slot index of st
        int jseg = 0;
        int js_base = 0;
        bool ok = true;
        for (int gp = 0; ok && gp < 4 * L; ++gp) {
            int r0, r1;
            block_range(p, gp, c, r0, r1);
            if (r0 >= r1) continue;
            const int KT = p.kind[gp & 3].k_tiles;
            for (int seg_start = r0; ok && seg_start < r1; ++jseg) {
                const int seg_end = min(r1, (seg_start / KT + 1) * KT);
                const int b = (p.nacc == 2) ? (jseg & 1) : 0;
                const uint32_t phb = (p.nacc == 2) ? ((jseg >> 1) & 1) : (jseg & 1);
                int r = seg_start + ((seg_start - r0 - mq) & 1);
                const int first = r;
                const bool oka = mbar_wait(smem_u32(&ctrl->accempty[b]), phb ^ 1, abort, p.err, kErrMma);
                if (!__all_sync(kAllOnes, oka)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (mq * p.nacc + b) * p.npad;
                for (; r < seg_end; r += 2) {
                    const int js = js_base + ((r - r0) >> 1);
                    st.advance(js - js_cur, S);
                    js_cur = js;
                    const int s = st.idx;
                    const bool okw = mbar_wait(smem_u32(&ctrl->afull[s]), st.phase, abort, p.err, kErrMma) &&
                                     mbar_wait(smem_u32(&ctrl->xfull[s]), st.phase, abort, p.err, kErrMma);
                    if (!__all_sync(kAllOnes, okw)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    mma4_bf16_ts_elect(d, a_slot(0, mq) + static_cast<uint32_t>(s) * astep,
                                       bdesc0 + static_cast<uint64_t>(s) * bstep, idesc, r != first ? 1u : 0u,
                                       smem_u32(&ctrl->empty[s]));
                    mma_issued = js + 1;
                }
                if (!ok) break;
                if (first < seg_end)
                    mma_commit_elect(smem_u32(&ctrl->accfull[b]));
                else
                    mbar_arrive_elect(smem_u32(&ctrl->accfull[b]));
                seg_start = seg_end;
            }
            if (!ok) break;
            const int nslots = (r1 - r0 + 1) >> 1;
            if (mq == 1 && ((r1 - r0) & 1)) {
                // the phase's last slot holds one record: release it for issuer 1 once it is full
                const int js = js_base + nslots - 1;
                st.advance(js - js_cur, S);
                js_cur = js;
                const bool okw = mbar_wait(smem_u32(&ctrl->afull[st.idx]), st.phase, abort, p.err, kErrMma);
                if (!__all_sync(kAllOnes, okw)) break;
                mbar_arrive_elect(smem_u32(&ctrl->empty[st.idx]));
            }
            js_base += nslots;
        }
    } else if (warp == kWEscape) {
        // ------------------------------------------------- record and escape feeder (warp-wide)
        // Per slot, as soon as its shared-memory slot is free (rfree): the summary of the slot's
        // index words (how many, how many belong to its first record, where they start) for the
        // decode groups, and the bulk copies of the slot's records, of its index words and of its
        // window bases, all counted on the slot's full barrier. Lane l holds rec_esc_off[wbase + l] (cur) and [wbase + 32 + l] (nxt) of the
        // current phase's tensor, so the offsets are loaded 32 at a time, ahead of use.
        SlotIt it = start;
        RingS st;
        int wgp = -1, wbase = 0;
        uint32_t cur = 0, nxt = 0;
        const uint32_t *offs = nullptr, *words = nullptr;
        const uint8_t *bases = nullptr, *recs = nullptr;
        int R = 0, KT = 1, ftile = 0, fkt = 0;  // tile and k tile of the slot's first record
        auto load_off = [&](int i) -> uint32_t { return (i <= R) ? __ldg(offs + i) : 0u; };
        while (!it.end(p)) {
            if (it.gp != wgp) {  // the phase's buffers, loaded once per phase
                wgp = it.gp;
                const STensor &T = p.t[wgp >> 2][wgp & 3];
                offs = T.rec_esc_off;
                words = T.rec_esc;
                bases = T.base_exp;
                recs = T.records;
                R = p.kind[wgp & 3].R;
                KT = p.kind[wgp & 3].k_tiles;
                wbase = it.r;
                cur = load_off(wbase + lane);
                nxt = load_off(wbase + 32 + lane);
                ftile = it.r / KT;
                fkt = it.r - ftile * KT;
            }
            while (it.r + it.nr >= wbase + 64) {
                wbase += 32;
                cur = nxt;
                nxt = load_off(wbase + 32 + lane);
            }
            auto off_of = [&](int i) -> uint32_t {
                const int dd = i - wbase;
                const uint32_t a = __shfl_sync(kAllOnes, cur, dd & 31);
                const uint32_t b2 = __shfl_sync(kAllOnes, nxt, dd & 31);
                return dd < 32 ? a : b2;
            };
            const uint32_t lo = off_of(it.r), mid = off_of(it.r + 1), hi = off_of(it.r + it.nr);
            const int tile0 = ftile;
            const bool new_tile = it.nr == 2 && fkt + 1 == KT;  // the second record starts the next tile
            const int s = st.idx;
            const bool ok = mbar_wait(smem_u32(&ctrl->rfree[s]), st.phase ^ 1, abort, p.err, kErrEscape);
            if (!__all_sync(kAllOnes, ok)) break;
            const uint32_t fb = smem_u32(&ctrl->full[s]);
            const uint32_t cnt = hi - lo;
            const bool staged = cnt > 0 && cnt <= static_cast<uint32_t>(kEscCapS);
            if (lane == 0) {
                ctrl->esc_info[s] = make_uint2(staged || cnt == 0 ? cnt : (cnt | 0x80000000u),
                                               (it.nr == 2) ? mid - lo : cnt);
                ctrl->esc_ptr[s] = words + lo;
                ctrl->slot_nr[s] = it.nr;
                ctrl->slot_en1[s] = new_tile ? kTileN : 0;
            }
            __syncwarp();
            // the slot's records, its escape words (when they fit) and the window bases of its
            // records' tiles
            const uint32_t en_bytes = new_tile ? 2u * kTileN : kTileN;
            const uint32_t rbytes = static_cast<uint32_t>(it.nr) * kRecordBytes;
            mbar_arrive_expect_tx_elect(fb, rbytes + (staged ? cnt * 4 : 0u) + en_bytes);
            bulk_g2s_elect(smem_u32(stage_rec(s, 0)), recs + static_cast<size_t>(it.r) * kRecordBytes, rbytes, fb);
            if (staged) bulk_g2s_elect(smem_u32(stage_esc(s)), words + lo, cnt * 4, fb);
            bulk_g2s_elect(smem_u32(stage_en(s)), bases + static_cast<size_t>(tile0) * kTileN, new_tile ? 2u * kTileN : kTileN,
                           fb);
            fkt += it.nr;
            while (fkt >= KT) {
                fkt -= KT;
                ++ftile;
            }
            it.next(p, c);
            st.advance(1, Sm);
            issued = it.js;
        }
    } else if (warp >= kWDec0) {
        // ---------------------------------------------------------------- decode groups
        // Group g decodes slots g, g + 3, g + 6, ... of the block's sequence: each thread its row
        // of each record (view bytes and plane B -> 32 bf16x2 words), stored to its tensor-memory
        // lane, then the warp's escapes patched in tensor memory; then the shared-memory slot is
        // handed back to the feeder (rfree) and the tensor-memory slot to the MMAs (afull).
        // Everything a slot needs besides its records (record count, window bases, escape words)
        // was staged by the escape feeder.
        const int g = (warp - kWDec0) >> 2;
        const int qw = warp & 3;
        const int nl = 32 * qw + lane;
        const uint32_t m3 = p.m3, m15 = p.m15;
        const uint32_t lanes = static_cast<uint32_t>(32 * qw) << 16;
        const int nslots = ctrl->nslots;
        RingS st;
        st.advance(g, S);
        uint32_t wa[32], wb[32];
        auto decode_record = [&](int s, int q, uint32_t base2, uint32_t (&w)[32]) {
            const uint8_t *rec = stage_rec(s, q);
            const uint4 v0 = lds128(rec + 0 * 2048 + 16 * nl);
            const uint4 v1 = lds128(rec + 1 * 2048 + 16 * nl);
            const uint4 v2 = lds128(rec + 2 * 2048 + 16 * nl);
            const uint4 v3 = lds128(rec + 3 * 2048 + 16 * nl);
            const uint4 b0 = lds128(rec + kViewBytes + 16 * nl);
            const uint4 b1 = lds128(rec + kViewBytes + 2048 + 16 * nl);
            decode_chunk16<false, 0>(v0, b0, base2, w, m3, m15);
            decode_chunk16<false, 1>(v1, b0, base2, w + 8, m3, m15);
            decode_chunk16<false, 0>(v2, b1, base2, w + 16, m3, m15);
            decode_chunk16<false, 1>(v3, b1, base2, w + 24, m3, m15);
        };
        // the escapes of record q of shared-memory slot m (decoded into tensor-memory slot s) that
        // fall in this warp's 32 rows: read the entry's column, let the owner lane overwrite its
        // half, write the column back
        auto patch_record = [&](int m, int s, int q, uint2 ei) {
            const uint32_t hdr = ei.x;
            const uint32_t total = hdr & 0x7FFFFFFFu;
            const uint32_t split = ei.y;
            const uint32_t sg0 = (q == 0) ? 0u : split, sg1 = (q == 0) ? split : total;
            if (sg1 <= sg0) return;
            const uint32_t *seg = ((hdr >> 31) ? ctrl->esc_ptr[m] : reinterpret_cast<const uint32_t *>(stage_esc(m))) + sg0;
            const uint32_t i_hi = seg[qw];
            const uint32_t tbase = a_slot(s, q) + lanes;
            for (uint32_t i = (qw == 0) ? 0u : seg[qw - 1]; i < i_hi; ++i) {
                const uint32_t ent = seg[4 + i];
                const uint32_t taddr = tbase + ((ent & 63u) >> 1);
                const uint32_t old = tmem_ld_32x32b_x1(taddr);
                tmem_wait_ld();
                const uint32_t nv = (ent & 1u) ? ((old & 0x0000FFFFu) | (ent & 0xFFFF0000u))
                                               : ((old & 0xFFFF0000u) | (ent >> 16));
                tmem_st_32x32b_x1(taddr, lane == static_cast<int>((ent >> 6) & 31u) ? nv : old);
                tmem_wait_st();
            }
        };
        // A slot's shared-memory position (m) and tensor-memory position (s) come from rings of
        // different sizes. When a ring's size is not a multiple of the group count, consecutive
        // uses of a position go to different groups: before waiting for a use of the position,
        // wait until the previous group's use of it is complete (rfree, afull), so that a parity
        // wait cannot be satisfied by a phase two uses old.
        const bool shared_m = (Sm % kDecGroupsS) != 0, shared_s = (S % kDecGroupsS) != 0;
        RingS rm;
        rm.advance(g, Sm);
        for (int js = g; js < nslots; js += kDecGroupsS) {
            const int s = st.idx, m = rm.idx;
            if (shared_m) {
                const bool ok_prev = mbar_wait(smem_u32(&ctrl->rfree[m]), rm.phase ^ 1, abort, p.err, kErrDecode);
                if (!__all_sync(kAllOnes, ok_prev)) break;
            }
            const bool ok_full = mbar_wait(smem_u32(&ctrl->full[m]), rm.phase, abort, p.err, kErrDecode);
            if (!__all_sync(kAllOnes, ok_full)) break;
            const int nr = ctrl->slot_nr[m];
            const uint8_t *en = stage_en(m);
            decode_record(m, 0, base2_of(en[nl]), wa);
            // the tensor-memory slot is free once the MMAs of its previous use have completed
            if (shared_s) {
                const bool ok_prev = mbar_wait(smem_u32(&ctrl->afull[s]), st.phase ^ 1, abort, p.err, kErrDecode);
                if (!__all_sync(kAllOnes, ok_prev)) break;
            }
            const bool ok_empty = mbar_wait(smem_u32(&ctrl->empty[s]), st.phase ^ 1, abort, p.err, kErrDecode);
            if (!__all_sync(kAllOnes, ok_empty)) break;
            tc_fence_after();
            tmem_st_32x32b_x32(a_slot(s, 0) + lanes, wa);
            if (nr == 2) {
                decode_record(m, 1, base2_of(en[ctrl->slot_en1[m] + nl]), wb);
                tmem_st_32x32b_x32(a_slot(s, 1) + lanes, wb);
            }
            tmem_wait_st();
            const uint2 ei = ctrl->esc_info[m];
            if (ei.x != 0) {
                patch_record(m, s, 0, ei);
                if (nr == 2) patch_record(m, s, 1, ei);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&ctrl->afull[s]));
            mbar_arrive(smem_u32(&ctrl->rfree[m]));
            st.advance(kDecGroupsS, S);
            rm.advance(kDecGroupsS, Sm);
        }
    } else {
        // ---------------------------------------------------------------- epilogue + glue (4 warps)
        const int qw = warp & 3;
        const int nl = 32 * qw + lane;
        const int et = threadIdx.x - kWEpi0 * 32;  // 0..127
        bool dead = false;
        int jseg = 0;
        // one thread waits for a phase to have completed on every block, then the four warps go on
        auto wait_phase = [&](int ph) {
            bool ok = true;
            if (et == 0 && !dead) ok = wait_count(p.done + ph, Gu, abort, p.err, kErrEpilogue);
            dead = named_bar_or(kEpiBarS, 128, !ok) || dead;
        };
        // the epilogue's stores of a phase are complete; count this block for the phase (a release
        // increment after the block barrier: the four warps' stores are visible to whoever
        // acquires the count)
        auto signal_phase = [&](int ph) {
            named_bar_sync(kEpiBarS, 128);
            if (et == 0) {
                if (ph < kPhasesPerLayer * L) {
                    red_release_gpu(p.done + ph, 1u);
                } else if (atom_add_acq_rel_gpu(p.done + ph, 1u) == Gu - 1) {
                    // every block has passed every wait of this launch: leave the counters zeroed
                    for (int i = 0; i <= kPhasesPerLayer * L; ++i) p.done[i] = 0;
                    for (int i = 0; i < kKinds * p.max_tiles; ++i) p.tile_cnt[i] = 0;
                }
            }
        };
        // ---- row normalisation phase: x = bf16(h / rms(h)); units (row, column chunk) over blocks
        auto rms_phase = [&](uint16_t *x) {
            constexpr int kRF = 4;  // 16-byte loads in flight per thread
            const int H = p.H, H4 = H >> 2;
            const int C = p.rms_chunks;
            const int Q4 = (H4 + C - 1) / C;
            if (H4 <= 128 * kRowF4) {
                // The row fits in the unit (thread et holds float4 et + 128 t, the array in local
                // memory): one round of loads, then the same arithmetic in the same order as the
                // passes below, in rolled loops. The phase runs once per layer from a cold
                // instruction cache, and unrolled it took longer to fetch than to execute.
                for (int u = c; !dead && u < M * C; u += G) {
                    const int m = u / C, ch = u % C;
                    const float4 *h4 = reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(m) * H);
                    float4 v[kRowF4];
#pragma unroll
                    for (int t = 0; t < kRowF4; ++t)
                        v[t] = (et + 128 * t < H4) ? __ldcg(h4 + et + 128 * t) : make_float4(0.f, 0.f, 0.f, 0.f);
                    float amax = 0.f;
#pragma unroll 1
                    for (int t = 0; t < kRowF4; ++t)
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[t].x), fabsf(v[t].y)), fmaxf(fabsf(v[t].z), fabsf(v[t].w))));
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kAllOnes, amax, off));
                    if (lane == 0) ctrl->red_max[qw] = amax;
                    named_bar_sync(kEpiBarS, 128);
                    const float bmax = fmaxf(fmaxf(ctrl->red_max[0], ctrl->red_max[1]), fmaxf(ctrl->red_max[2], ctrl->red_max[3]));
                    uint16_t *xr = x + static_cast<size_t>(m) * H;
                    const int i_lo = ch * Q4, i_hi = min((ch + 1) * Q4, H4);
                    if (bmax == 0.f) {  // an all-zero row
                        for (int i = i_lo + et; i < i_hi; i += 128) __stcg(reinterpret_cast<uint2 *>(xr) + i, make_uint2(0u, 0u));
                        named_bar_sync(kEpiBarS, 128);
                        continue;
                    }
                    const int e = ilogbf(bmax) + 1;  // |h| * 2^-e < 1
                    // four independent pair sums (one per 32-bit lane of the 16-byte words), so the
                    // dependent chain is a quarter as long; then combined in a fixed order
                    F2 a4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 1
                    for (int t = 0; t < kRowF4; ++t) {
                        const float q[4] = {scale_pow2(v[t].x, -e), scale_pow2(v[t].y, -e), scale_pow2(v[t].z, -e),
                                            scale_pow2(v[t].w, -e)};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float pp = __fmul_rn(q[j], q[j]);
                            a4[j] = f2_add(a4[j], F2{pp, __fmaf_rn(q[j], q[j], -pp)});
                        }
                    }
                    F2 acc = f2_add(f2_add(a4[0], a4[1]), f2_add(a4[2], a4[3]));
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        acc = f2_add(acc, F2{__shfl_xor_sync(kAllOnes, acc.hi, off), __shfl_xor_sync(kAllOnes, acc.lo, off)});
                    if (lane == 0) ctrl->red_sum[qw] = acc;
                    named_bar_sync(kEpiBarS, 128);
                    if (et == 0) {
                        F2 tt = ctrl->red_sum[0];
                        for (int i = 1; i < 4; ++i) tt = f2_add(tt, ctrl->red_sum[i]);
                        ctrl->scale = rms_scale(tt, p.inv_h);
                    }
                    named_bar_sync(kEpiBarS, 128);
                    const float yh = ctrl->scale.yh, yl = ctrl->scale.yl;
                    // this thread's words in the unit's chunk: t with i_lo <= et + 128 t < i_hi
                    const int t_lo = (i_lo > et) ? (i_lo - et + 127) / 128 : 0;
#pragma unroll 1
                    for (int t = t_lo; t < kRowF4; ++t) {
                        const int i = et + 128 * t;
                        if (i >= i_hi) break;
                        {
                            uint2 out;
                            out.x = static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[t].x, -e), yh, yl)) |
                                    (static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[t].y, -e), yh, yl)) << 16);
                            out.y = static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[t].z, -e), yh, yl)) |
                                    (static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[t].w, -e), yh, yl)) << 16);
                            __stcg(reinterpret_cast<uint2 *>(xr) + i, out);
                        }
                    }
                    named_bar_sync(kEpiBarS, 128);  // ctrl's scratch is free for the next unit
                }
                return;
            }
            for (int u = c; !dead && u < M * C; u += G) {
                const int m = u / C, ch = u % C;
                const float4 *h4 = reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(m) * H);
                // pass 1: the largest |h| of the row
                float amax = 0.f;
                for (int base = et; base < H4; base += 128 * kRF) {
                    float4 v[kRF];
#pragma unroll
                    for (int j = 0; j < kRF; ++j)
                        v[j] = (base + 128 * j < H4) ? __ldcg(h4 + base + 128 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kRF; ++j)
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kAllOnes, amax, off));
                if (lane == 0) ctrl->red_max[qw] = amax;
                named_bar_sync(kEpiBarS, 128);
                const float bmax = fmaxf(fmaxf(ctrl->red_max[0], ctrl->red_max[1]), fmaxf(ctrl->red_max[2], ctrl->red_max[3]));
                uint16_t *xr = x + static_cast<size_t>(m) * H;
                const int i_lo = ch * Q4, i_hi = min((ch + 1) * Q4, H4);
                if (bmax == 0.f) {  // an all-zero row
                    for (int i = i_lo + et; i < i_hi; i += 128) __stcg(reinterpret_cast<uint2 *>(xr) + i, make_uint2(0u, 0u));
                    named_bar_sync(kEpiBarS, 128);
                    continue;
                }
                const int e = ilogbf(bmax) + 1;  // |h| * 2^-e < 1
                // pass 2: the sum of squares of h * 2^-e in fp32 pairs (the row is in L2 by now)
                F2 acc = {0.f, 0.f};
                for (int base = et; base < H4; base += 128 * kRF) {
                    float4 v[kRF];
#pragma unroll
                    for (int j = 0; j < kRF; ++j)
                        v[j] = (base + 128 * j < H4) ? __ldcg(h4 + base + 128 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kRF; ++j) {
                        const float q[4] = {scale_pow2(v[j].x, -e), scale_pow2(v[j].y, -e), scale_pow2(v[j].z, -e),
                                            scale_pow2(v[j].w, -e)};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float pp = __fmul_rn(q[t], q[t]);
                            acc = f2_add(acc, F2{pp, __fmaf_rn(q[t], q[t], -pp)});
                        }
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    acc = f2_add(acc, F2{__shfl_xor_sync(kAllOnes, acc.hi, off), __shfl_xor_sync(kAllOnes, acc.lo, off)});
                if (lane == 0) ctrl->red_sum[qw] = acc;
                named_bar_sync(kEpiBarS, 128);
                if (et == 0) {
                    F2 t = ctrl->red_sum[0];
                    for (int i = 1; i < 4; ++i) t = f2_add(t, ctrl->red_sum[i]);
                    ctrl->scale = rms_scale(t, p.inv_h);
                }
                named_bar_sync(kEpiBarS, 128);
                const float yh = ctrl->scale.yh, yl = ctrl->scale.yl;
                for (int base = i_lo + et; base < i_hi; base += 128 * kRF) {
                    float4 v[kRF];
#pragma unroll
                    for (int j = 0; j < kRF; ++j)
                        v[j] = (base + 128 * j < i_hi) ? __ldcg(h4 + base + 128 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kRF; ++j) {
                        if (base + 128 * j < i_hi) {
                            uint2 out;
                            out.x = static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[j].x, -e), yh, yl)) |
                                    (static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[j].y, -e), yh, yl)) << 16);
                            out.y = static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[j].z, -e), yh, yl)) |
                                    (static_cast<uint32_t>(bf16_mul_rne(scale_pow2(v[j].w, -e), yh, yl)) << 16);
                            __stcg(reinterpret_cast<uint2 *>(xr) + base + 128 * j, out);
                        }
                    }
                }
                named_bar_sync(kEpiBarS, 128);  // ctrl's scratch is free for the next unit
            }
        };
        // ---- the outputs of 16 rows m0.. of tile `tile` of a GEMM of kind k (f: this thread's column)
        auto finalize = [&](int k, int tile, int m0, const float (&f)[16]) {
            if (k == kKindGu) {
                // lanes 0-63 of the tile hold gate rows, lanes 64-127 the matching up rows: the up
                // half goes through shared memory to the thread of its gate row
                if (qw >= 2) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) xchg[i * 64 + (nl - 64)] = f[i];
                }
                named_bar_sync(kEpiBarS, 128);
                if (qw < 2) {
                    const int n = tile * 64 + nl;  // column of p
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (m0 + i < M && n < p.F) {
                            const float prod = __fmul_rn(f[i], xchg[i * 64 + nl]);
                            __stcg(reinterpret_cast<unsigned short *>(p.pg) + static_cast<size_t>(m0 + i) * p.F + n,
                                   __bfloat16_as_ushort(__float2bfloat16_rn(prod)));
                        }
                    }
                }
                named_bar_sync(kEpiBarS, 128);
                return;
            }
            const int n = tile * kTileN + nl;
            if (n >= p.kind[k].N) return;
            if (k == kKindQkv) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (m0 + i < M)
                        __stcg(reinterpret_cast<unsigned short *>(p.qkv) + static_cast<size_t>(m0 + i) * p.Nqkv + n,
                               __bfloat16_as_ushort(__float2bfloat16_rn(f[i])));
            } else {  // o and down: one fp32 addition into h per element
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (m0 + i < M) {
                        float *hp = p.h + static_cast<size_t>(m0 + i) * p.H + n;
                        __stcg(hp, __ldcg(hp) + f[i]);
                    }
            }
        };
        // ---- one GEMM phase: this block's segments, in order
        auto gemm_phase_epi = [&](int gp) {
            int r0, r1;
            block_range(p, gp, c, r0, r1);
            const int k = gp & 3;
            const SKind &K = p.kind[k];
            const int KT = K.k_tiles, U = K.unit, units = K.R / K.unit;
            float *part_base = p.partials + static_cast<size_t>(gp & 1) * G * 2 * M * kTileN;
            auto bstart = [&](int cc) { return U * range_start_s(cc, units, K.grid); };
            auto part_of = [&](int cc, int tile) {
                const int sl = (bstart(cc) / KT == tile) ? 0 : 1;
                return part_base + (static_cast<size_t>(cc) * 2 + sl) * M * kTileN;
            };
            // split tiles of this phase whose sum this block shares (its first and last segment)
            int split_tile[2], split_lo[2], split_hi[2], nsplit = 0;
            for (int seg_start = r0; seg_start < r1; ++jseg) {
                const int tile = seg_start / KT;
                const int seg_end = min(r1, (tile + 1) * KT);
                const bool full = seg_start == tile * KT && seg_end == (tile + 1) * KT;
                const int b = (p.nacc == 2) ? (jseg & 1) : 0;
                const uint32_t phb = (p.nacc == 2) ? ((jseg >> 1) & 1) : (jseg & 1);
                const bool ok = !dead && mbar_wait(smem_u32(&ctrl->accfull[b]), phb, abort, p.err, kErrEpilogue);
                dead = named_bar_or(kEpiBarS, 128, !ok) || dead;
                const int c_lo = full ? c : owner_of_s((tile * KT) / U, units, K.grid);
                const int c_hi = full ? c : owner_of_s(((tile + 1) * KT - 1) / U, units, K.grid);
                float *part = part_of(c, tile);
                if (!dead) {
                    tc_fence_after();
                    const bool has0 = ((seg_start - r0) & 1) == 0 || seg_end - seg_start >= 2;
                    const bool has1 = ((seg_start - r0) & 1) == 1 || seg_end - seg_start >= 2;
                    const uint32_t ln = static_cast<uint32_t>(32 * qw) << 16;
                    const uint32_t t0 = tmem + ln + (0 * p.nacc + b) * p.npad;
                    const uint32_t t1 = tmem + ln + (1 * p.nacc + b) * p.npad;
#pragma unroll 1
                    for (int m0 = 0; m0 < M; m0 += 16) {
                        float f[16];
                        uint32_t v[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] = 0.f;
                        if (has0) {
                            tmem_ld_32x32b_x16(t0 + m0, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
                        }
                        if (has1) {
                            tmem_ld_32x32b_x16(t1 + m0, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) f[i] = has0 ? f[i] + __uint_as_float(v[i]) : __uint_as_float(v[i]);
                        }
                        if (full) {
                            finalize(k, tile, m0, f);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (m0 + i < M) __stcg(part + static_cast<size_t>(m0 + i) * kTileN + nl, f[i]);
                        }
                    }
                    tc_fence_before();
                }
                mbar_arrive(smem_u32(&ctrl->accempty[b]));
                if (!full && !dead && k != kKindGu) {
                    // publish the part; the tile's sum is formed after the block's last segment
                    named_bar_sync(kEpiBarS, 128);
                    if (et == 0) red_release_gpu(p.tile_cnt + k * p.max_tiles + tile, 1u);
                    split_tile[nsplit] = tile;
                    split_lo[nsplit] = c_lo;
                    split_hi[nsplit] = c_hi;
                    ++nsplit;
                } else if (!full && !dead) {
                    // gate|up split tile: whichever block publishes its part last sums all parts in
                    // block order (the product needs both halves of every row of the tile)
                    named_bar_sync(kEpiBarS, 128);
                    if (et == 0) {
                        const uint32_t old = atom_add_acq_rel_gpu(p.tile_cnt + k * p.max_tiles + tile, 1u);
                        ctrl->last = (old == static_cast<uint32_t>(c_hi - c_lo)) ? 1 : 0;
                    }
                    named_bar_sync(kEpiBarS, 128);
                    if (ctrl->last) {
#pragma unroll 1
                        for (int m0 = 0; m0 < M; m0 += 16) {
                            float f[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) f[i] = 0.f;
#pragma unroll 1
                            for (int cb = c_lo; cb <= c_hi; ++cb) {
                                const float *src = part_of(cb, tile);
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (m0 + i < M) f[i] += __ldcg(src + static_cast<size_t>(m0 + i) * kTileN + nl);
                            }
                            finalize(k, tile, m0, f);
                        }
                        if (et == 0) p.tile_cnt[k * p.max_tiles + tile] = 0;  // leave the workspace zeroed
                    }
                    named_bar_sync(kEpiBarS, 128);  // ctrl->last is read by every thread before it changes
                }
                seg_start = seg_end;
            }
            // Sums of the split tiles. Every block of a tile published its part above before it
            // waits here, so the waits cannot form a cycle. Once all parts are in (the tile's
            // counter grows by its block count in every layer), block c_lo + i sums the i-th of
            // the tile's c_hi - c_lo + 1 slices of 16-byte groups (row m, columns 4j..4j+3) over the
            // parts in increasing block order, the same additions in the same order as a single
            // summing block, and writes them out.
            const uint32_t layer1 = static_cast<uint32_t>((gp >> 2) + 1);
#pragma unroll 1
            for (int sidx = 0; sidx < nsplit && !dead; ++sidx) {
                const int tile = split_tile[sidx], c_lo = split_lo[sidx], c_hi = split_hi[sidx];
                const int np = c_hi - c_lo + 1;
                bool okc = true;
                if (et == 0)  // an acquire load of the count; the barrier below passes it to the block
                    okc = wait_count(p.tile_cnt + k * p.max_tiles + tile, layer1 * static_cast<uint32_t>(np), abort, p.err,
                                     kErrEpilogue);
                dead = named_bar_or(kEpiBarS, 128, !okc) || dead;
                if (dead) break;
                const int G4 = M * (kTileN / 4);
                const int g_lo = (c - c_lo) * G4 / np, g_hi = (c - c_lo + 1) * G4 / np;
                constexpr int kG = 2, kP = 4;  // groups per thread per round, parts per round of loads
#pragma unroll 1
                for (int g0 = g_lo + et; g0 < g_hi; g0 += 128 * kG) {
                    float4 acc[kG], hv[kG];
#pragma unroll
                    for (int q = 0; q < kG; ++q) {
                        acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                        const int g = g0 + 128 * q;
                        const int m = g / (kTileN / 4), n = tile * kTileN + 4 * (g % (kTileN / 4));
                        hv[q] = (k != kKindQkv && g < g_hi && n < K.N)
                                    ? __ldcg(reinterpret_cast<const float4 *>(p.h + static_cast<size_t>(m) * p.H + n))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll 1
                    for (int cb = c_lo; cb <= c_hi; cb += kP) {
                        float4 v[kP][kG];
#pragma unroll
                        for (int j = 0; j < kP; ++j) {
                            const float4 *src = reinterpret_cast<const float4 *>(part_of(min(cb + j, c_hi), tile));
#pragma unroll
                            for (int q = 0; q < kG; ++q)
                                v[j][q] = (cb + j <= c_hi && g0 + 128 * q < g_hi) ? __ldcg(src + g0 + 128 * q)
                                                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int j = 0; j < kP; ++j) {
                            if (cb + j > c_hi) break;
#pragma unroll
                            for (int q = 0; q < kG; ++q) {
                                acc[q].x += v[j][q].x;
                                acc[q].y += v[j][q].y;
                                acc[q].z += v[j][q].z;
                                acc[q].w += v[j][q].w;
                            }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kG; ++q) {
                        const int g = g0 + 128 * q;
                        if (g >= g_hi) break;
                        const int m = g / (kTileN / 4), n = tile * kTileN + 4 * (g % (kTileN / 4));
                        if (n >= K.N) continue;
                        if (k == kKindQkv) {
                            uint2 o;
                            o.x = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[q].x))) |
                                  (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[q].y))) << 16);
                            o.y = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[q].z))) |
                                  (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[q].w))) << 16);
                            __stcg(reinterpret_cast<uint2 *>(reinterpret_cast<unsigned short *>(p.qkv) +
                                                             static_cast<size_t>(m) * p.Nqkv + n), o);
                        } else {  // o and down: one fp32 addition into h per element
                            const float4 r = make_float4(hv[q].x + acc[q].x, hv[q].y + acc[q].y, hv[q].z + acc[q].z,
                                                         hv[q].w + acc[q].w);
                            __stcg(reinterpret_cast<float4 *>(p.h + static_cast<size_t>(m) * p.H + n), r);
                        }
                    }
                }
            }
        };
        for (int l = 0; l < L && !dead; ++l) {
            const int ph = kPhasesPerLayer * l;
            if (l > 0) wait_phase(ph - 1);  // h after the previous layer's down projection
            rms_phase(p.xa);
            signal_phase(ph);
            gemm_phase_epi(4 * l + kKindQkv);
            signal_phase(ph + 1);
            gemm_phase_epi(4 * l + kKindO);
            signal_phase(ph + 2);
            wait_phase(ph + 2);
            rms_phase(p.xm);
            signal_phase(ph + 3);
            gemm_phase_epi(4 * l + kKindGu);
            signal_phase(ph + 4);
            gemm_phase_epi(4 * l + kKindDown);
            signal_phase(ph + 5);
        }
        if (!dead) {
            wait_phase(kPhasesPerLayer * L - 1);
            rms_phase(p.x_out);
            signal_phase(kPhasesPerLayer * L);
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    // after an abort, let copies still in flight land before the block's shared memory is released
    if (warp == kWEscape && lane == 0 && ctrl->abort) {
        for (int js = (issued > Sm ? issued - Sm : 0); js < issued; ++js)
            if (!mbar_wait_drain(smem_u32(&ctrl->full[js % Sm]), (js / Sm) & 1)) atomicOr(p.err, kErrDrain);
    }
    if (warp == kWProducer && lane == 0 && ctrl->abort) {
        for (int js = (xissued > S ? xissued - S : 0); js < xissued; ++js)
            if (!mbar_wait_drain(smem_u32(&ctrl->xfull[js % S]), (js / S) & 1)) atomicOr(p.err, kErrDrain);
    }
    if ((warp == kWMma || warp == kWMma2) && mma_issued > 0) {
        const int mq = (warp == kWMma) ? 0 : 1;
        mma_commit_elect(smem_u32(&ctrl->drained[mq]));
        if (!mbar_wait_drain(smem_u32(&ctrl->drained[mq]), 0) && lane == 0) atomicOr(p.err, kErrDrain);
    }
    __syncthreads();
    if (warp == kWMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemColsS);
    }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

constexpr double kSplitSlack = 1.15;  // the work split of w12_gemm (whole tiles when they balance)
constexpr int64_t kMinRecs = 8;

struct StreamPlan {
    SKind kind[kKinds];
    int H, F, Nqkv, nq, npad, stages, rstages, nacc, acc_cols, G, sbytes, smem, rms_chunks, max_tiles;
    size_t off_err, off_done, off_tile, off_part, off_xa, off_xm, off_qkv, off_p, ws_bytes;
};

void split_of(const w12_tensor &t, int sms, SKind *k) {
    k->N = t.N;
    k->K = t.K;
    k->n_tiles = t.n_tiles;
    k->k_tiles = t.k_tiles;
    k->R = t.n_tiles * t.k_tiles;
    const int T = t.n_tiles;
    const int per = (T + sms - 1) / sms;
    if (static_cast<double>(per) * sms <= kSplitSlack * T) {
        k->grid = (T + per - 1) / per;
        k->unit = t.k_tiles;
    } else {
        const int64_t by_work = (k->R + kMinRecs - 1) / kMinRecs;
        k->grid = static_cast<int>(std::min<int64_t>({std::max<int64_t>(T, by_work), k->R, sms}));
        k->unit = 1;
    }
}

bool same_shape(const w12_tensor &a, const w12_tensor &b) { return a.N == b.N && a.K == b.K; }

w12_status plan_stream(const w12_stream_layer *layers, int n_layers, int M, int n_q, StreamPlan *P) {
    if (!layers || n_layers < 1 || n_layers > kMaxLayersS) return W12_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxMS) return W12_ERR_UNSUPPORTED_SHAPE;
    const w12_stream_layer &l0 = layers[0];
    for (int l = 0; l < n_layers; ++l) {
        const w12_stream_layer &ll = layers[l];
        W12_TRY(check_tensor(&ll.qkv));
        W12_TRY(check_tensor(&ll.o));
        W12_TRY(check_tensor(&ll.gate_up));
        W12_TRY(check_tensor(&ll.down));
        if (!same_shape(ll.qkv, l0.qkv) || !same_shape(ll.o, l0.o) || !same_shape(ll.gate_up, l0.gate_up) ||
            !same_shape(ll.down, l0.down))
            return W12_ERR_INVALID_ARG;
    }
    const int H = l0.qkv.K, F = l0.down.K, Nqkv = l0.qkv.N;
    if (l0.o.N != H || l0.gate_up.K != H || l0.down.N != H || l0.gate_up.N != 2 * F || l0.o.K != n_q)
        return W12_ERR_INVALID_ARG;
    if (n_q < 1 || n_q > Nqkv) return W12_ERR_INVALID_ARG;
    // every activation is read as whole 64-wide k slices, and each tile of gate|up pairs 64 gate
    // rows with 64 up rows
    if (H % kTileK || F % kTileK || n_q % kTileK || Nqkv % 8) return W12_ERR_UNSUPPORTED_SHAPE;
    int sms = 0;
    W12_TRY(require_device(&sms));
    split_of(l0.qkv, sms, &P->kind[kKindQkv]);
    split_of(l0.o, sms, &P->kind[kKindO]);
    split_of(l0.gate_up, sms, &P->kind[kKindGu]);
    split_of(l0.down, sms, &P->kind[kKindDown]);
    P->H = H;
    P->F = F;
    P->Nqkv = Nqkv;
    P->nq = n_q;
    P->G = sms;
    P->npad = (M + 15) / 16 * 16;
    // tensor-memory slots: what the accumulators leave of the 512 columns; each with its two
    // activation tiles (npad x 128 bytes, so every tile starts on a 128-byte-swizzle atom); then as
    // many shared-memory slots of copied records as the rest of shared memory holds
    P->sbytes = 2 * P->npad * 128;
    const int ctrl = static_cast<int>(align_up(kSCtrlBytes + kXchgBytes, 1024));
    P->nacc = 2;
    P->acc_cols = 2 * P->nacc * P->npad;
    const int stages = std::min(kMaxStagesS, (kTmemColsS - P->acc_cols) / (2 * kAColsS));
    const int rstages = std::min(kMaxRawS, (kSmemLimitS - 1024 - ctrl - stages * P->sbytes) / kRawBytes);
    if (stages < kDecGroupsS || rstages < kDecGroupsS) return W12_ERR_UNSUPPORTED_SHAPE;
    P->stages = stages;
    P->rstages = rstages;
    P->smem = 1024 + stages * P->sbytes + rstages * kRawBytes + ctrl;
    // row-normalisation units: (row, chunk of the row) spread over the blocks
    const int H4 = H / 4;
    // (every unit reads its whole row for the statistics and writes its chunk: spreading the
    // writes over more blocks shortens the phase while blocks are left over)
    P->rms_chunks = std::max(1, std::min(std::max(1, sms / M), (H4 + 7) / 8));
    P->max_tiles = 0;
    for (const SKind &k : P->kind) P->max_tiles = std::max(P->max_tiles, k.n_tiles);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    P->off_err = take(16);
    P->off_done = take(sizeof(uint32_t) * (kPhasesPerLayer * n_layers + 1));
    P->off_tile = take(sizeof(uint32_t) * kKinds * P->max_tiles);
    P->off_part = take(sizeof(float) * 2 * static_cast<size_t>(sms) * 2 * M * kTileN);
    P->off_xa = take(2 * static_cast<size_t>(M) * H);
    P->off_xm = take(2 * static_cast<size_t>(M) * H);
    P->off_qkv = take(2 * static_cast<size_t>(M) * Nqkv);
    P->off_p = take(2 * static_cast<size_t>(M) * F);
    P->ws_bytes = off;
    return W12_OK;
}

// x as [M rows, K] bf16 with rows ldx elements apart: one 64-wide k slice (map), two
// consecutive slices (map2), 128-byte swizzle, rows padded to npad by the copy's zero fill
w12_status x_maps(const uint16_t *x, int K, int ldx, int M, int npad, CUtensorMap *map, CUtensorMap *map2) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return W12_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
    const cuuint32_t box[2] = {kTileK, static_cast<cuuint32_t>(npad)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return W12_ERR_INVALID_ARG;
    const cuuint64_t dims3[3] = {static_cast<cuuint64_t>(kTileK), static_cast<cuuint64_t>(M),
                                 static_cast<cuuint64_t>(K / kTileK)};
    const cuuint64_t strides3[2] = {static_cast<cuuint64_t>(ldx) * 2, static_cast<cuuint64_t>(kTileK) * 2};
    const cuuint32_t box3[3] = {kTileK, static_cast<cuuint32_t>(npad), 2};
    const cuuint32_t estr3[3] = {1, 1, 1};
    if (enc(map2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(x), dims3, strides3, box3, estr3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return W12_ERR_INVALID_ARG;
    return W12_OK;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" w12_status w12_stream_workspace_size(const w12_stream_layer *layers, int n_layers, int M, int n_q,
                                                size_t *bytes) {
    if (!bytes) return W12_ERR_INVALID_ARG;
    StreamPlan P{};
    W12_TRY(plan_stream(layers, n_layers, M, n_q, &P));
    *bytes = P.ws_bytes;
    return W12_OK;
}

extern "C" w12_status w12_stream_buffers(const w12_stream_layer *layers, int n_layers, int M, int n_q,
                                         size_t offsets[4]) {
    if (!offsets) return W12_ERR_INVALID_ARG;
    StreamPlan P{};
    W12_TRY(plan_stream(layers, n_layers, M, n_q, &P));
    offsets[0] = P.off_xa;
    offsets[1] = P.off_qkv;
    offsets[2] = P.off_xm;
    offsets[3] = P.off_p;
    return W12_OK;
}

extern "C" w12_status w12_stream_step_ex(const w12_stream_layer *layers, int n_layers, int M, int n_q, float *h,
                                         uint16_t *x_out, void *workspace, size_t workspace_bytes, unsigned flags,
                                         w12_stream_t stream) {
    if (!h || !x_out || !workspace) return W12_ERR_INVALID_ARG;
    if (flags & ~static_cast<unsigned>(W12_LAUNCH_TEST_STALL)) return W12_ERR_INVALID_ARG;
    if (!aligned16(h) || (reinterpret_cast<uintptr_t>(x_out) & 7u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return W12_ERR_INVALID_ARG;
    StreamPlan P{};
    W12_TRY(plan_stream(layers, n_layers, M, n_q, &P));
    if (workspace_bytes < P.ws_bytes) return W12_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SParams *sp = new (std::nothrow) SParams();
    if (!sp) return W12_ERR_CUDA;
    SParams &p = *sp;
    p.L = n_layers;
    p.M = M;
    p.npad = P.npad;
    p.stages = P.stages;
    p.rstages = P.rstages;
    p.nacc = P.nacc;
    p.acc_cols = P.acc_cols;
    p.G = P.G;
    p.H = P.H;
    p.F = P.F;
    p.Nqkv = P.Nqkv;
    p.rms_chunks = P.rms_chunks;
    p.inv_h = f2_of(1.0 / static_cast<double>(P.H));
    p.sbytes = P.sbytes;
    p.h = h;
    p.xa = reinterpret_cast<uint16_t *>(ws + P.off_xa);
    p.xm = reinterpret_cast<uint16_t *>(ws + P.off_xm);
    p.qkv = reinterpret_cast<uint16_t *>(ws + P.off_qkv);
    p.pg = reinterpret_cast<uint16_t *>(ws + P.off_p);
    p.x_out = x_out;
    p.partials = reinterpret_cast<float *>(ws + P.off_part);
    p.tile_cnt = reinterpret_cast<uint32_t *>(ws + P.off_tile);
    p.max_tiles = P.max_tiles;
    p.done = reinterpret_cast<uint32_t *>(ws + P.off_done);
    p.err = reinterpret_cast<int *>(ws + P.off_err);
    p.m3 = 8u;
    p.m15 = 32768u;
    p.test_stall = (flags & W12_LAUNCH_TEST_STALL) ? 1 : 0;
    for (int k = 0; k < kKinds; ++k) p.kind[k] = P.kind[k];
    for (int l = 0; l < n_layers; ++l) {
        const w12_tensor *ts[kKinds] = {&layers[l].qkv, &layers[l].o, &layers[l].gate_up, &layers[l].down};
        for (int k = 0; k < kKinds; ++k)
            p.t[l][k] = STensor{ts[k]->records, ts[k]->base_exp, ts[k]->rec_esc_off, ts[k]->rec_esc};
    }
    w12_status st = W12_OK;
    // the activations each kind reads: x (normalised rows), the q columns of q|k|v in place, the
    // normalised MLP input, the gate-up product
    CUtensorMap xm[kKinds], xm2[kKinds];
    if (st == W12_OK) st = x_maps(p.xa, P.H, P.H, M, P.npad, &xm[kKindQkv], &xm2[kKindQkv]);
    if (st == W12_OK) st = x_maps(p.qkv, P.nq, P.Nqkv, M, P.npad, &xm[kKindO], &xm2[kKindO]);
    if (st == W12_OK) st = x_maps(p.xm, P.H, P.H, M, P.npad, &xm[kKindGu], &xm2[kKindGu]);
    if (st == W12_OK) st = x_maps(p.pg, P.F, P.F, M, P.npad, &xm[kKindDown], &xm2[kKindDown]);
    if (st == W12_OK) {
        static std::atomic<uint64_t> smem_set{0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) st = W12_ERR_CUDA;
        const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
        if (st == W12_OK && (!bit || !(smem_set.load(std::memory_order_acquire) & bit))) {
            if (cudaFuncSetAttribute(w12_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimitS) !=
                cudaSuccess)
                st = W12_ERR_CUDA;
            else
                smem_set.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    if (st == W12_OK) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(P.G));
        cfg.blockDim = dim3(kThreadsS);
        cfg.dynamicSmemBytes = static_cast<size_t>(P.smem);
        cfg.stream = reinterpret_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;  // every block resident: they wait on one another
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, w12_stream_kernel, xm[0], xm2[0], xm[1], xm2[1], xm[2], xm2[2], xm[3], xm2[3], p) !=
            cudaSuccess)
            st = W12_ERR_CUDA;
    }
    delete sp;
    return st;
}

extern "C" w12_status w12_stream_step(const w12_stream_layer *layers, int n_layers, int M, int n_q, float *h,
                                      uint16_t *x_out, void *workspace, size_t workspace_bytes, w12_stream_t stream) {
    return w12_stream_step_ex(layers, n_layers, M, n_q, h, x_out, workspace, workspace_bytes, 0u, stream);
}

extern "C" w12_status w12_stream_interleave(const uint16_t *gate, const uint16_t *up, int ffn, int hidden,
                                            uint16_t *gate_up, w12_stream_t stream) {
    if (!gate || !up || !gate_up || ffn < 1 || hidden < 1) return W12_ERR_INVALID_ARG;
    if (ffn % 64) return W12_ERR_UNSUPPORTED_SHAPE;
    // rows [128 i, 128 i + 64) of gate_up = gate rows [64 i, 64 i + 64), the next 64 = up's
    const size_t row = static_cast<size_t>(hidden) * 2, blk = 64 * row;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpy2DAsync(gate_up, 2 * blk, gate, blk, blk, static_cast<size_t>(ffn / 64), cudaMemcpyDeviceToDevice,
                          st) != cudaSuccess)
        return W12_ERR_CUDA;
    if (cudaMemcpy2DAsync(reinterpret_cast<uint8_t *>(gate_up) + blk, 2 * blk, up, blk, blk,
                          static_cast<size_t>(ffn / 64), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return W12_ERR_CUDA;
    return W12_OK;
}

