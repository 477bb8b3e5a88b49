// a3/a4/a5 — the skinny W12 GEMM on 5th-generation tensor cores (tcgen05, sm_103a).
//
// SpecPilot §4.1 and Fig. 5b: the weights are expanded from W12 on chip, inside the GEMM, where
// the expansion overlaps the weight stream from memory; the k range is shared out between
// blocks whose parts are added in an order that never changes, so results repeat bit for bit;
// §6.3 and App. E: it is bound by weight bytes at 1-32 rows; §4.3: the Q pass reads only the
// nested 8-bit view; §2.1: greedy verification takes the row argmax.
//
// Design on GB300 (one persistent block per SM, 8 + 4*G warps with G = W12_DECODE_GROUPS decode
// groups, 20 warps by default). Work moves through a ring of
// `stages` slots; a slot holds `rps` consecutive records (2 for up to 64 rows, else 1) with
// their activation tiles and escape entries in shared memory, plus one 32-column tensor-memory
// buffer per record for the decoded weights. Each slot has three barriers: full (copies
// landed), afull (decoded weights stored) and empty (the MMAs that read it completed).
//   warp 0       producer: one bulk copy of the slot's records (contiguous in memory), one
//                128B-swizzled TMA box of the activations' k-slice per record
//   warps 1, 3   warp 1 allocates tensor memory; one elected thread of each issues tcgen05.mma
//                (M=128 weight rows from tensor memory, N = rows of x padded to 16 from shared
//                memory, K=16): warp 1 for the first record of every slot, warp 3 for the second,
//                each into an fp32 accumulator of its own
//   warp 2       escape feeder: bulk-copies the slot's escape entries next to its records
//   warps 4-7    epilogue: tensor memory -> registers; y, split-K partials or the row argmax
//   warps 8-     G decode groups of 4 warps, taking slots in turn: each thread owns one weight
//                row of a record, turns its 64 view bytes + 32 plane-B bytes into 32 bf16x2
//                words, patches its escapes and stores them into its tensor-memory lane (the
//                MMA's A operand)
// The single-thread roles wait on a barrier once per slot, not once per record: a barrier
// round trip costs a few hundred cycles, comparable to the HBM time of one 12 KB record.
// Work split: the R = n_tiles*k_tiles records are cut into `grid` contiguous, equal ranges
// (stream-K). A tile covered by several blocks is finished by whichever arrives last, summing
// the blocks' fp32 partials in increasing block order: no float atomics, bitwise reproducible.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstddef>
#include <mutex>

#include "w12_internal.cuh"


namespace w12 {
namespace {

#ifndef W12_DECODE_GROUPS
#define W12_DECODE_GROUPS 3
#endif
constexpr int kDecGroups = W12_DECODE_GROUPS;     // decode groups of 4 warps (one per lane quarter)
constexpr int kThreads = 32 * (8 + 4 * kDecGroups);
static_assert(kDecGroups >= 1 && kDecGroups <= 4, "one to four decode groups");
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpEscape = 2;
constexpr int kWarpMma2 = 3;  // second MMA issuer (the second record of each slot)
constexpr int kWarpEpi0 = 4;
constexpr int kWarpDec0 = 8;
constexpr int kEscCap = 128;       // index words staged per slot; more -> read from global
constexpr int kStageBufs = 2;      // tensor-store staging buffers per epilogue warp
constexpr int kACols = 32;         // tensor-memory columns of one decoded record (64 bf16/lane)
constexpr int kMaxStages = 8;
constexpr int kMaxM = W12_MAX_M;
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 232448;       // opt-in maximum per block
constexpr int kSmemFloor = 120 * 1024;   // keeps one block per SM
constexpr int kEpiBar = 1;               // named barrier of the 128 epilogue threads
// Whole tiles per block are used when the busiest block then has at most this factor of the
// average work: up to 15% imbalance costs less than splitting tiles and summing the partials
// at the end (measured on the 136-tile MLP projection on 152 SMs).
#ifndef W12_TILE_SPLIT_SLACK
#define W12_TILE_SPLIT_SLACK 1.15
#endif
constexpr double kTileSplitSlack = W12_TILE_SPLIT_SLACK;
// Stream-K blocks get at least this many records (measured on the 8-tile k/v projections: 152
// blocks of 4 records -> 80 blocks of 8: 21 us -> 8 us at M=32, the split partials halved)
#ifndef W12_MIN_RECORDS_PER_BLOCK
#define W12_MIN_RECORDS_PER_BLOCK 8
#endif
constexpr int64_t kMinRecordsPerBlock = W12_MIN_RECORDS_PER_BLOCK;

struct Ctrl {
    uint64_t full[kMaxStages], afull[kMaxStages], empty[kMaxStages], xfull[kMaxStages];
    uint64_t accfull[2], accempty[2];
    uint64_t done[2];
    // per slot: x = index words of the slot (bit 31: too many to stage, read from global),
    // y = words that belong to the slot's first record; one 8-byte load for the decode warps
    uint2 esc_info[kMaxStages];
    uint32_t esc_src[kMaxStages];    // index of the slot's first word in the global index
    uint32_t tmem_base;
    int abort;
    int fix;          // block-wide flag of the final argmax merge
    int mode[2];      // how a split tile ends (by segment parity)
    int last[2];      // this block published last and sums the tile (by segment parity)
    int pre;          // the last segment's other block had published before its MMAs completed
};

// After the control block, 128-byte aligned, the epilogue's scratch: in the argmax variants the
// per-warp top-2 of each row (4 x M float4) and the block's running top-2 (M float4); in the
// GEMM variants the staging buffers of the tensor stores of y (4 warps x 2 x 16 x 32 words).
constexpr size_t kCtrlBytes = (sizeof(Ctrl) + 127) / 128 * 128;
constexpr size_t kStagingBytes = 4 * kStageBufs * 16 * 32 * 4;
// the argmax variants need their top-2 records, the GEMM variants the tensor-store staging
// (tensor stores of y measured faster than plain stores at every row count: at M=192 plain
// stores and the sixth ring slot they free cost 6 us a launch)
constexpr size_t scratch_bytes(int M, bool argmax) {
    return argmax ? 80 * static_cast<size_t>(M) : kStagingBytes;
}

struct Params {
    const uint8_t *records;
    const uint8_t *base_exp;
    const uint32_t *rec_esc_off;
    const uint32_t *rec_esc;
    int N, K, M, n_tiles, k_tiles, npad, stages, rps, nacc, acc_cols, grid;
    int unit;  // records per unit of the work split: 1 (stream-K) or k_tiles (whole tiles)
    int overlap;  // launched as a programmatic dependent launch (W12_LAUNCH_OVERLAP)
    int y_tma;    // y is written by tiled tensor stores through ymap
    int y_accum;  // W12_LAUNCH_ACCUMULATE: y (fp32) += the result instead of y = the result
    int v_tma;    // Q view: a slot's two record views arrive by one tiled copy through vmap
    int xhalf;    // more than 256 rows: rows per activation box and per MMA (npad / 2), else 0
    const float *row_scale;  // INT8 / INT6 copy: per-channel scale, [n_tiles * 128]
    int *run_flag;           // if set, the launch does nothing unless *run_flag != 0 (then clears it)
    int x_pair;   // xmap2 loads the k-slices of two consecutive records in one copy
    int test_stall;  // W12_LAUNCH_TEST_STALL: the producer fills only the first slot
    uint32_t m3, m15;  // 8 and 32768: decode multipliers, given at run time (see decode_pair)
    int R;  // records: n_tiles * k_tiles (< 2^22)
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

// Record counts fit in 32 bits with room to spare (R <= 2^21 since N*K <= 2^31, and G <= 256),
// so block ranges use 32-bit arithmetic: a 64-bit division is a long software routine.
__device__ __forceinline__ int range_start(int c, int R, int G) {
    return static_cast<int>(static_cast<uint32_t>(c) * static_cast<uint32_t>(R) / static_cast<uint32_t>(G));
}
// the block whose range holds record i
__device__ __forceinline__ int owner_of(int i, int R, int G) {
    return static_cast<int>((static_cast<uint32_t>(i + 1) * G + R - 1) / static_cast<uint32_t>(R)) - 1;
}

// Position in a ring of `size` slots: index and the parity of its phase. Advanced
// incrementally so no per-record integer division is needed.
struct Ring {
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

// One halving step of the 16-row warp top-2 below: of rows [0, K) the lane keeps the upper half
// if (lane & O), else the lower half, merges in its partner's (lane ^ O) copy of those rows and
// stores them compacted at [0, K/2).
template <int K, int O>
__device__ __forceinline__ void top2_halve(float (&v1)[16], int (&i1)[16], float (&v2)[16], int lane) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int j = 0; j < K / 2; ++j) {
        float kv1 = up ? v1[j + K / 2] : v1[j], kv2 = up ? v2[j + K / 2] : v2[j];
        int ki1 = up ? i1[j + K / 2] : i1[j];
        const float gv1 = up ? v1[j] : v1[j + K / 2], gv2 = up ? v2[j] : v2[j + K / 2];
        const int gi1 = up ? i1[j] : i1[j + K / 2];
        const float rv1 = __shfl_xor_sync(0xFFFFFFFFu, gv1, O);
        const int ri1 = __shfl_xor_sync(0xFFFFFFFFu, gi1, O);
        const float rv2 = __shfl_xor_sync(0xFFFFFFFFu, gv2, O);
        top2_merge(kv1, ki1, kv2, rv1, ri1, rv2);
        v1[j] = kv1;
        i1[j] = ki1;
        v2[j] = kv2;
    }
}

// Top-2 over the warp's 32 columns of each of 16 rows, lane l holding column l of every row
// (v1 = value, i1 = its index, v2 = -inf on entry). Recursive halving: after the steps on lane
// bits 4..1 lane l holds row l >> 1 over the 16 lanes that share those bits; one exchange with
// lane l ^ 1 completes it. 15 row exchanges instead of 16 five-step reductions.
__device__ __forceinline__ void warp_top2_rows16(float (&v1)[16], int (&i1)[16], float (&v2)[16], int lane) {
    top2_halve<16, 16>(v1, i1, v2, lane);
    top2_halve<8, 8>(v1, i1, v2, lane);
    top2_halve<4, 4>(v1, i1, v2, lane);
    top2_halve<2, 2>(v1, i1, v2, lane);
    const float rv1 = __shfl_xor_sync(0xFFFFFFFFu, v1[0], 1);
    const int ri1 = __shfl_xor_sync(0xFFFFFFFFu, i1[0], 1);
    const float rv2 = __shfl_xor_sync(0xFFFFFFFFu, v2[0], 1);
    top2_merge(v1[0], i1[0], v2[0], rv1, ri1, rv2);
}

// kPack: 0 = W12 records; 8 = the INT8 copy (8 KB records of sign-magnitude codes); 6 = the
// INT6 copy (6 KB records of offset codes in two planes). The copies have no escapes, and each
// output channel's accumulator is multiplied by its row scale.
template <bool kQView, bool kArgmax, int kPack = 0>
__global__ void __launch_bounds__(kThreads, 1)
w12_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap xmap2,
                const __grid_constant__ CUtensorMap ymap, const __grid_constant__ CUtensorMap vmap, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a conditional launch (the certified head's fallback) that is not needed ends here, before
    // any barrier, copy or tensor memory is touched; the flag was written by an earlier kernel
    // on the stream, which has completed (this launch is stream-ordered)
    if (p.run_flag && *reinterpret_cast<volatile int *>(p.run_flag) == 0) return;
    // the next grid on the stream may start as soon as SMs free up; it waits for this grid's
    // completion itself before it reads activations or its workspace
    grid_launch_dependents();

    const int S = p.stages, RPS = p.rps;
    const int xbytes = p.npad * 128;
    constexpr bool kCopy = kPack != 0;  // a separate low-precision copy (INT8 or INT6)
    static_assert(kPack == 0 || kPack == 6 || kPack == 8, "W12 records, the INT8 or the INT6 copy");
    static_assert(!kCopy || kQView, "the copies are read like a view: no plane B, no escapes");
    constexpr int rbytes = (kPack == 6) ? kQ6RecordBytes : (kQView ? kViewBytes : kRecordBytes);
    constexpr int ebytes = kQView ? 0 : kEscCap * 4;
    // distance between records in memory
    constexpr int gstride = (kPack == 6) ? kQ6RecordBytes : (kCopy ? kViewBytes : kRecordBytes);
    // A slot's records arrive by one copy: whole records as one contiguous range; for the Q view
    // the two records' views by one tiled copy that skips the B planes between them (vmap), else
    // the range from the first record's view to the end of the last one's.
    const bool vtma = kQView && p.v_tma;
    // shared-memory distance between records
    const int rstride = (kPack == 6) ? kQ6RecordBytes : ((vtma || kCopy) ? kViewBytes : kRecordBytes);
    const int recs_bytes = (RPS - 1) * rstride + rbytes;
    const int sbytes = RPS * xbytes + recs_bytes + ebytes;
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + S * sbytes);
    uint8_t *scratch = reinterpret_cast<uint8_t *>(ctrl) + kCtrlBytes;
    float4 *wtop = reinterpret_cast<float4 *>(scratch);          // [4][M]
    float4 *ctop = reinterpret_cast<float4 *>(scratch) + 4 * p.M;  // [M]
    auto stage_x = [&](int s, int q) { return smem + s * sbytes + q * xbytes; };
    auto stage_rec = [&](int s, int q) { return smem + s * sbytes + RPS * xbytes + q * rstride; };
    auto stage_esc = [&](int s) { return smem + s * sbytes + RPS * xbytes + recs_bytes; };

    const int c = blockIdx.x;
    const int R = p.R, G = p.grid, KT = p.k_tiles, U = p.unit;
    // block cc's range starts at record block_start(cc); owner(i) is the block holding record i
    auto block_start = [&](int cc) { return U * range_start(cc, R / U, G); };
    auto owner = [&](int i) { return owner_of(i / U, R / U, G); };
    const int r0 = block_start(c), r1 = block_start(c + 1);
    const int nrec = r1 - r0;
    const int nst = (nrec + RPS - 1) / RPS;  // slots this block fills

    int issued = 0;   // producer: slots whose records were handed to the copy engine; mma: slots issued
    int xissued = 0;  // producer: slots whose activation tiles were handed to the copy engine
    // producer state: its slot ring, the k tile of its next record, the next record's bytes
    Ring pst;
    int pkt = 0;
    const uint8_t *psrc = nullptr;
    // The records of a slot (full barrier, with the escape entries) and its activation tiles
    // (xfull barrier) arrive separately: records are weights, which no earlier kernel writes,
    // so they may be fetched and decoded before the previous grid on the stream has finished;
    // x and the workspace may not be touched before that (grid_dependency_wait).
    auto produce_rec = [&](int js) {  // ring slot pst.idx gets the records of slot js
        const int s = pst.idx;
        const int nr = min(RPS, nrec - js * RPS);
        const uint32_t fb = smem_u32(&ctrl->full[s]);
        if (vtma) {
            // the box always spans two records; past the last record it reads zeros, and a
            // record past this block's range is read but not decoded
            mbar_arrive_expect_tx_elect(fb, 2 * kViewBytes);
            tma_3d_g2s_elect(smem_u32(stage_rec(s, 0)), &vmap, 0, 0, r0 + js * 2, fb);
        } else {
            const uint32_t bytes = (nr - 1) * gstride + rbytes;  // consecutive records are contiguous
            mbar_arrive_expect_tx_elect(fb, bytes);
            bulk_g2s_elect(smem_u32(stage_rec(s, 0)), psrc, bytes, fb);
        }
        psrc += nr * gstride;
        issued = js + 1;
        pst.advance(1, S);
    };
    auto produce_x = [&](int js, int s) {  // ring slot s gets the activation tiles of slot js
        const int nr = min(RPS, nrec - js * RPS);
        const uint32_t xb = smem_u32(&ctrl->xfull[s]);
        mbar_arrive_expect_tx_elect(xb, nr * xbytes);
        if (p.x_pair && nr == 2 && pkt + 1 < p.k_tiles) {
            // both records in one k tile pair: slices pkt and pkt+1 land as two adjacent tiles
            tma_3d_g2s_elect(smem_u32(stage_x(s, 0)), &xmap2, 0, 0, pkt, xb);
            pkt += 2;
            if (pkt == p.k_tiles) pkt = 0;
        } else {
            for (int q = 0; q < nr; ++q) {
                tma_2d_g2s_elect(smem_u32(stage_x(s, q)), &xmap, pkt * kTileK, 0, xb);
                // above 256 rows the tile arrives as two boxes of xhalf rows
                if (p.xhalf) tma_2d_g2s_elect(smem_u32(stage_x(s, q) + p.xhalf * 128), &xmap, pkt * kTileK, p.xhalf, xb);
                if (++pkt == p.k_tiles) pkt = 0;
            }
        }
        xissued = js + 1;
    };

    if (warp == kWarpProducer) {
        // the producer initialises the barriers and starts the first slot's copies before the
        // block-wide barrier, so their HBM latency overlaps the rest of the set-up; the other
        // slots follow right after the barrier (issuing all of them here would hold every
        // other warp at the barrier while the copy engine takes them in)
        if (lane == 0) {
            for (int s = 0; s < S; ++s) {
                mbar_init(smem_u32(&ctrl->full[s]), kQView ? 1 : 2);
                mbar_init(smem_u32(&ctrl->afull[s]), 128);
                mbar_init(smem_u32(&ctrl->empty[s]), RPS);  // one commit per MMA issuer
                mbar_init(smem_u32(&ctrl->xfull[s]), 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&ctrl->accfull[b]), RPS);
                mbar_init(smem_u32(&ctrl->accempty[b]), 128);
            }
            mbar_init(smem_u32(&ctrl->done[0]), 1);
            mbar_init(smem_u32(&ctrl->done[1]), 1);
            ctrl->abort = 0;
            ctrl->fix = 0;
            fence_barrier_init();
            prefetch_tensormap(&xmap);
            prefetch_tensormap(&xmap2);
            if (vtma) prefetch_tensormap(&vmap);
        }
        __syncwarp();
        pkt = r0 % KT;
        psrc = p.records + static_cast<size_t>(r0) * gstride;
        if (nst > 0) produce_rec(0);
    }
    // escape feeder: lane l holds rec_esc_off[r0 + base + l] (cur) and [r0 + base + 32 + l]
    // (nxt); the first loads start here so their latency also overlaps the set-up
    auto esc_load = [&](int b0) -> uint32_t {
        const int i = r0 + b0 + lane;
        return (i <= R) ? __ldg(p.rec_esc_off + i) : 0u;
    };
    uint32_t esc_cur = 0, esc_nxt = 0;
    if (!kQView && warp == kWarpEscape) {
        esc_cur = esc_load(0);
        esc_nxt = esc_load(32);
    }
    // decode threads: their row's E_n for the block's first two tiles, requested before the
    // set-up barrier so that these loads are not queued behind the first slots' record copies
    const int en_row = 32 * (warp & 3) + lane;
    auto en_load = [&](int tile) -> uint32_t {
        return (tile < p.n_tiles) ? static_cast<uint32_t>(__ldg(p.base_exp + tile * kTileN + en_row)) : 0u;
    };
    int en_tile = r0 / KT;
    uint32_t en_cur = 0, en_nxt = 0;
    if (!kCopy && warp >= kWarpDec0) {
        en_cur = en_load(en_tile);
        en_nxt = en_load(en_tile + 1);
    }
    if (kArgmax) {
        for (int m = threadIdx.x; m < p.M; m += kThreads)
            ctop[m] = make_float4(-INFINITY, __int_as_float(0x7FFFFFFF), -INFINITY, 0.f);
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    auto a_slot = [&](int s, int q) { return tmem + p.acc_cols + (s * RPS + q) * kACols; };
    volatile int *abort = &ctrl->abort;

    if (warp == kWarpProducer) {
        // ---------------------------------------------------------------- producer (warp-wide)
        // The copy engine serves requests in order, so a slot's activation tiles queued behind
        // the records of every later slot would hold its MMAs back by several microseconds.
        // Plain launch: each slot's records, then its tiles. Overlapped launch: the records of
        // every free slot first (they may load while the previous grid finishes), then the tiles
        // once it has (by then those record copies have drained).
        // the first S slots start out free; under the test hook only the first is filled, so
        // the block's bounded waits run out
        const int n0 = p.test_stall ? min(1, nst) : min(S, nst);
        if (p.overlap) {
            for (int js = 1; js < n0; ++js) produce_rec(js);
            grid_dependency_wait();  // x may be the previous grid's output
            for (int js = 0; js < n0; ++js) produce_x(js, js);
        } else {
            if (n0 > 0) produce_x(0, 0);
            for (int js = 1; js < n0; ++js) {
                produce_rec(js);
                produce_x(js, js);
            }
        }
        for (int js = n0; !p.test_stall && js < nst; ++js) {
            const int s = pst.idx;
            const bool ok = mbar_wait(smem_u32(&ctrl->empty[s]), pst.phase ^ 1, abort, p.err, kErrProducer);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            produce_rec(js);
            produce_x(js, s);
        }
    } else if (warp == kWarpMma || (warp == kWarpMma2 && RPS == 2)) {
        // ---------------------------------------------------------------- MMA issuers (warp-wide)
        // With two records per slot, issuer mq = 0 (warp 1) takes the first record of every slot
        // and issuer mq = 1 (warp 3) the second, each into an accumulator of its own: a single
        // warp cannot issue the MMAs of both records in the time the copy engine brings them.
        // Per segment each issuer overwrites its accumulator with its first record, adds the
        // rest, and commits (or, without a record in the segment, just arrives on) accfull.
        const int mq = (warp == kWarpMma) ? 0 : 1;
        const uint32_t idesc = idesc_bf16_f32(128, p.xhalf ? p.xhalf : p.npad);
        const uint64_t bhalf = static_cast<uint64_t>((p.xhalf * 128) >> 4);  // descriptor step to row xhalf
        // the slot's operands: its activation tile for this issuer (B, by descriptor; the
        // descriptor's start-address field moves by sbytes / 16 per slot) and the issuer's
        // decoded record (A, in tensor memory)
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(stage_x(0, mq)));
        const uint64_t bstep = static_cast<uint64_t>(sbytes >> 4);
        const uint32_t a0 = a_slot(0, mq);
        const uint32_t astep = static_cast<uint32_t>(RPS * kACols);
        Ring st;
        int js_next = 0;  // ring position of st: the slot of this issuer's next record
        int jseg = 0;
        bool ok = true;
        for (int seg_start = r0; ok && seg_start < r1; ++jseg) {
            const int seg_end = min(r1, (seg_start / KT + 1) * KT);
            const int b = (p.nacc == 2) ? (jseg & 1) : 0;
            const uint32_t phb = (p.nacc == 2) ? ((jseg >> 1) & 1) : (jseg & 1);
            // this issuer's records r in [seg_start, seg_end) have (r - r0) % RPS == mq
            int r = seg_start + ((seg_start - r0 - mq) & (RPS - 1));
            const int first = r;
            const bool oka = mbar_wait(smem_u32(&ctrl->accempty[b]), phb ^ 1, abort, p.err, kErrMma);
            if (!__all_sync(0xFFFFFFFFu, oka)) break;
            tc_fence_after();
            const uint32_t d = tmem + (mq * p.nacc + b) * p.npad;
            for (; r < seg_end; r += RPS) {
                const int js = (r - r0) >> (RPS - 1);  // RPS is 1 or 2
                st.advance(js - js_next, S);
                js_next = js;
                const int s = st.idx;
                const bool okw = mbar_wait(smem_u32(&ctrl->afull[s]), st.phase, abort, p.err, kErrMma) &&
                                 mbar_wait(smem_u32(&ctrl->xfull[s]), st.phase, abort, p.err, kErrMma);
                if (!__all_sync(0xFFFFFFFFu, okw)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the issuer's first MMA of a segment overwrites its accumulator; the rest add
                if (p.xhalf)
                    mma4x2_bf16_ts_elect(d, a0 + static_cast<uint32_t>(s) * astep, bdesc0 + static_cast<uint64_t>(s) * bstep,
                                         bhalf, static_cast<uint32_t>(p.xhalf), idesc, r != first ? 1u : 0u,
                                         smem_u32(&ctrl->empty[s]));
                else
                    mma4_bf16_ts_elect(d, a0 + static_cast<uint32_t>(s) * astep, bdesc0 + static_cast<uint64_t>(s) * bstep,
                                       idesc, r != first ? 1u : 0u, smem_u32(&ctrl->empty[s]));
                issued = js + 1;
            }
            if (!ok) break;
            if (first < seg_end)
                mma_commit_elect(smem_u32(&ctrl->accfull[b]));
            else
                mbar_arrive_elect(smem_u32(&ctrl->accfull[b]));
            seg_start = seg_end;
        }
    } else if (warp == kWarpEscape) {
        // ---------------------------------------------------------------- escape feeder (warp-wide)
        if (!kQView) {
            int base = 0;
            uint32_t cur = esc_cur, nxt = esc_nxt;
            auto off_of = [&](int i) -> uint32_t {  // requires i - base in [0, 64)
                const int dd = i - base;
                const uint32_t a = __shfl_sync(0xFFFFFFFFu, cur, dd & 31);
                const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, nxt, dd & 31);
                return dd < 32 ? a : b2;
            };
            Ring st;
            for (int js = 0; js < nst; ++js, st.advance(1, S)) {
                const int first = js * RPS;
                const int nr = min(RPS, nrec - first);
                if (first >= base + 32) {
                    base += 32;
                    cur = nxt;
                    nxt = esc_load(base + 32);
                }
                const uint32_t lo = off_of(first);
                const uint32_t mid = off_of(first + 1);
                const uint32_t hi = off_of(first + nr);
                const int s = st.idx;
                const bool ok = mbar_wait(smem_u32(&ctrl->empty[s]), st.phase ^ 1, abort, p.err, kErrEscape);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                const uint32_t fb = smem_u32(&ctrl->full[s]);
                const uint32_t cnt = hi - lo;
                if (lane == 0) {
                    ctrl->esc_info[s] = make_uint2((cnt <= static_cast<uint32_t>(kEscCap)) ? cnt : (cnt | 0x80000000u),
                                                   (nr == 2) ? mid - lo : cnt);
                    ctrl->esc_src[s] = lo;
                }
                __syncwarp();  // the header stores come before the arrive that publishes them
                if (cnt == 0 || cnt > static_cast<uint32_t>(kEscCap)) {
                    mbar_arrive_elect(fb);
                } else {
                    mbar_arrive_expect_tx_elect(fb, cnt * 4);
                    bulk_g2s_elect(smem_u32(stage_esc(s)), p.rec_esc + lo, cnt * 4, fb);
                }
            }
        }
    } else if (warp >= kWarpDec0) {
        // ---------------------------------------------------------------- decode groups
        // Group g decodes every record of slots g, g + G, g + 2G, ... (G = kDecGroups). With
        // two records per slot, a thread decodes its row of the first record, stores it to tensor
        // memory, and decodes the second while that store is in flight; one wait covers both.
        const int g = (warp - kWarpDec0) >> 2;
        const int qw = warp & 3;
        const int nl = 32 * qw + lane;
        const uint32_t m3 = p.m3, m15 = p.m15;
        // this row's E_n for tile en_tile (en_cur) and the tile after it (en_nxt): moving to the
        // next tile takes the value already loaded and starts the load of the one after
        auto base2_for = [&](int tile) -> uint32_t {
            while (en_tile < tile) {
                en_cur = en_nxt;
                ++en_tile;
                en_nxt = en_load(en_tile + 1);
            }
            return base2_of(static_cast<int>(en_cur));
        };
        // decode this thread's row of record q of slot s into w (escapes patched)
        auto decode_record = [&](int s, int q, uint32_t base2, uint32_t (&w)[32]) {
            const uint8_t *rec = stage_rec(s, q);
            if constexpr (kPack == 6) {
                // plane L words 0-3 (groups 0, 1) and 4-7 (groups 2, 3), then plane T words 0-3
                const uint4 l0 = lds128(rec + 16 * nl);
                const uint4 l1 = lds128(rec + 2048 + 16 * nl);
                const uint4 tw = lds128(rec + 4096 + 16 * nl);
                decode_q6_group16(l0.x, l0.y, tw.x, w);
                decode_q6_group16(l0.z, l0.w, tw.y, w + 8);
                decode_q6_group16(l1.x, l1.y, tw.z, w + 16);
                decode_q6_group16(l1.z, l1.w, tw.w, w + 24);
                return;
            }
            const uint4 v0 = lds128(rec + 0 * 2048 + 16 * nl);
            const uint4 v1 = lds128(rec + 1 * 2048 + 16 * nl);
            const uint4 v2 = lds128(rec + 2 * 2048 + 16 * nl);
            const uint4 v3 = lds128(rec + 3 * 2048 + 16 * nl);
            if constexpr (kPack == 8) {
                decode_q8_chunk16(v0, w);
                decode_q8_chunk16(v1, w + 8);
                decode_q8_chunk16(v2, w + 16);
                decode_q8_chunk16(v3, w + 24);
                return;
            }
            if (kQView) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                decode_chunk16<true, 0>(v0, z, base2, w, m3, m15);
                decode_chunk16<true, 1>(v1, z, base2, w + 8, m3, m15);
                decode_chunk16<true, 0>(v2, z, base2, w + 16, m3, m15);
                decode_chunk16<true, 1>(v3, z, base2, w + 24, m3, m15);
                return;
            }
            const uint4 b0 = lds128(rec + kViewBytes + 16 * nl);
            const uint4 b1 = lds128(rec + kViewBytes + 2048 + 16 * nl);
            decode_chunk16<false, 0>(v0, b0, base2, w, m3, m15);
            decode_chunk16<false, 1>(v1, b0, base2, w + 8, m3, m15);
            decode_chunk16<false, 0>(v2, b1, base2, w + 16, m3, m15);
            decode_chunk16<false, 1>(v3, b1, base2, w + 24, m3, m15);
        };
        // Restore the escapes of record q of slot s that fall in this warp's 32 rows, in tensor
        // memory after the decoded record was stored there: read the entry's column, let the
        // owner lane overwrite its half, write the column back. One entry per round trip (a
        // few instructions each; the typical warp has 0-3). The segment header gives the
        // warp's entry range directly; every lane reads the same entry (a broadcast), so the
        // control flow is warp-uniform.
        auto patch_record = [&](int s, int q, uint2 ei) {
            const uint32_t hdr = ei.x;
            const uint32_t total = hdr & 0x7FFFFFFFu;
            const uint32_t split = ei.y;
            const uint32_t sg0 = (q == 0) ? 0u : split, sg1 = (q == 0) ? split : total;
            if (sg1 <= sg0) return;
            const uint32_t *seg = ((hdr >> 31) ? p.rec_esc + ctrl->esc_src[s]
                                               : reinterpret_cast<const uint32_t *>(stage_esc(s))) + sg0;
            const uint32_t i_hi = seg[qw];
            const uint32_t tbase = a_slot(s, q) + (static_cast<uint32_t>(32 * qw) << 16);
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
        int js = g;
        Ring st;
        st.advance(js, S);
        int tile = (r0 + js * RPS) / KT;  // tile and k tile of the slot's first record
        int kt = (r0 + js * RPS) % KT;
        uint32_t wa[32], wb[32];
        // A parity wait cannot tell phase u from phase u - 2. When G divides S, a slot's uses all
        // fall to one group, which has seen use u - 1 complete before it waits for use u. When it
        // does not, the previous use belongs to another group and its copies may land after this
        // group's last slot: wait until that use was decoded (afull phase u - 1; afull cannot
        // lag further, since the in-order MMA issuer consumed use u - 2 before the producer
        // issued anything this group has decoded) so the full wait below sees phase u itself.
        const bool shared_slots = (S % kDecGroups) != 0;
        for (; js < nst; js += kDecGroups) {
            const int s = st.idx;
            if (shared_slots) {
                const bool ok_prev = mbar_wait(smem_u32(&ctrl->afull[s]), st.phase ^ 1, abort, p.err, kErrDecode);
                if (!__all_sync(0xFFFFFFFFu, ok_prev)) break;
            }
            const bool ok_full = mbar_wait(smem_u32(&ctrl->full[s]), st.phase, abort, p.err, kErrDecode);
            if (!__all_sync(0xFFFFFFFFu, ok_full)) break;
            const int nr = min(RPS, nrec - js * RPS);
            // the slot's tensor-memory buffers are free: the producer refilled this slot only
            // after the MMAs that last read it completed
            decode_record(s, 0, kCopy ? 0u : base2_for(tile), wa);
            tc_fence_after();
            tmem_st_32x32b_x32(a_slot(s, 0) + (static_cast<uint32_t>(32 * qw) << 16), wa);
            if (nr == 2) {
                const int tile1 = (kt + 1 == p.k_tiles) ? tile + 1 : tile;
                decode_record(s, 1, kCopy ? 0u : base2_for(tile1), wb);
                tmem_st_32x32b_x32(a_slot(s, 1) + (static_cast<uint32_t>(32 * qw) << 16), wb);
            }
            tmem_wait_st();
            if (!kQView) {
                const uint2 ei = ctrl->esc_info[s];
                if (ei.x != 0) {  // the slot has index words
                    patch_record(s, 0, ei);
                    if (nr == 2) patch_record(s, 1, ei);
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&ctrl->afull[s]));
            st.advance(kDecGroups, S);
            kt += RPS * kDecGroups;
            while (kt >= p.k_tiles) {
                kt -= p.k_tiles;
                ++tile;
            }
        }
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
        // ---------------------------------------------------------------- epilogue
        // A segment that covers a whole tile is written directly. A tile split between blocks
        // is summed in increasing block order by the block that finishes it: if every other
        // block has already published its partial (the usual case for a block's last segment),
        // this block adds them to its own values straight from tensor memory; otherwise it
        // publishes its partial and whichever block publishes last sums all of them. Both
        // routes add the same values in the same order.
        const int qw = warp & 3;
        const int nl = 32 * qw + lane;
        const int et = threadIdx.x - kWarpEpi0 * 32;  // 0..127
        const int M = p.M;
        bool dead = false;
        grid_dependency_wait();  // the workspace and y may still be in use by the previous grid
        int jseg = 0;
        int r = r0;
        auto store_y = [&](int m, int n, float f) {
            if (p.y_bf16)
                reinterpret_cast<__nv_bfloat16 *>(p.y)[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(f);
            else if (p.y_accum)  // this thread alone writes the element in this launch
                reinterpret_cast<float *>(p.y)[static_cast<size_t>(m) * p.N + n] += f;
            else
                reinterpret_cast<float *>(p.y)[static_cast<size_t>(m) * p.N + n] = f;
        };
        // one output value of row m (warp-uniform call): y, or this warp's top-2 of the row
        auto emit = [&](int m, int n, float f) {
            if (kArgmax) {
                float v1 = (n < p.N && !isnan(f)) ? f : -INFINITY, v2 = -INFINITY;
                int i1 = n;
                warp_top2(v1, i1, v2);
                if (lane == 0) wtop[qw * M + m] = make_float4(v1, __int_as_float(i1), v2, 0.f);
            } else if (n < p.N) {
                store_y(m, n, f);
            }
        };
        // Rows m0..m0+15 of this thread's column leave for y (or the argmax) or for this block's
        // partial. y goes out through the copy engine when the tensor map allows it (p.y_tma):
        // each warp stages its 16 x 32 block in shared memory (two buffers, the argmax scratch
        // area) and one lane issues a tiled tensor store, which writes only the elements inside
        // y. The warps then need not wait for the stores to drain, which under the weight stream
        // of the blocks still running takes microseconds per chunk. Partial sums, read back by
        // another block, are stored directly, one value per row.
        int ybuf = 0;
        auto put_rows = [&](int m0, int tile, const float (&f)[16], float *part) {
          if constexpr (!kArgmax) {
            if (!part && p.y_tma) {
                const int esz = p.y_bf16 ? 2 : 4;
                uint8_t *stg = scratch + (qw * kStageBufs + ybuf) * 16 * 32 * esz;
                ybuf = (ybuf + 1) % kStageBufs;
                if (lane == 0) bulk_wait_group_read<kStageBufs - 1>();  // the store that last read this buffer
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (p.y_bf16)
                        reinterpret_cast<__nv_bfloat16 *>(stg)[i * 32 + lane] = __float2bfloat16_rn(f[i]);
                    else
                        reinterpret_cast<float *>(stg)[i * 32 + lane] = f[i];
                }
                fence_proxy_async_shared();
                __syncwarp();
                // a box that starts at or beyond column N writes nothing: not issued
                if (lane == 0 && tile * kTileN + 32 * qw < p.N) {
                    if (p.y_accum)  // each element of y gets exactly one addition per launch
                        tma_2d_s2g_add(&ymap, tile * kTileN + 32 * qw, m0, smem_u32(stg));
                    else
                        tma_2d_s2g(&ymap, tile * kTileN + 32 * qw, m0, smem_u32(stg));
                    bulk_commit_group();
                }
                return;
            }
          }
          if constexpr (kArgmax) {
            if (!part) {
                // this warp's top-2 of each of the 16 rows, into wtop[qw * M + m]
                const int n = tile * kTileN + nl;
                float v1[16], v2[16];
                int i1[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v1[i] = (n < p.N && !isnan(f[i])) ? f[i] : -INFINITY;
                    i1[i] = n;
                    v2[i] = -INFINITY;
                }
                warp_top2_rows16(v1, i1, v2, lane);
                const int m = m0 + (lane >> 1);
                if ((lane & 1) == 0 && m < M) wtop[qw * M + m] = make_float4(v1[0], __int_as_float(i1[0]), v2[0], 0.f);
                return;
            }
          }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (m0 + i >= M) break;
                if (part)
                    part[static_cast<size_t>(m0 + i) * kTileN + nl] = f[i];
                else
                    emit(m0 + i, tile * kTileN + nl, f[i]);
            }
        };
        // the INT8 and INT6 copies: a block's accumulator values are multiplied by their channel's
        // row scale as they leave tensor memory, so partials, their sums and y all carry the scale
        // once
        auto scale_rows = [&](int tile, float (&f)[16]) {
            if constexpr (kCopy) {
                const float sc = p.row_scale[tile * kTileN + nl];
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] *= sc;
            }
        };
        auto partial_of = [&](int cc, int tile, int m) {  // block cc's partial of tile
            const int sl = (block_start(cc) / KT == tile) ? 0 : 1;
            return p.partials + ((static_cast<size_t>(cc) * 2 + sl) * M + m) * kTileN + nl;
        };
        while (r < r1) {
            const int tile = r / KT;
            const int seg_start = r, seg_end = min(r1, (tile + 1) * KT);
            r = seg_end;
            const bool full = seg_start == tile * KT && seg_end == (tile + 1) * KT;
            const int par = jseg & 1;
            const int slot = (jseg == 0) ? 0 : 1;
            const int b = (p.nacc == 2) ? (jseg & 1) : 0;
            const uint32_t phb = (p.nacc == 2) ? ((jseg >> 1) & 1) : (jseg & 1);
            ++jseg;
            const int c_lo = full ? c : owner(tile * KT);
            const int c_hi = full ? c : owner((tile + 1) * KT - 1);
            // 0: whole tile here; 1: publish a partial; 2: sum here from the published partials
            int mode = 0;
            // A block's last segment ends the kernel for it. When its tile has one other block
            // and that block has already published (the usual case: the other block had the
            // tile at the start of its range), fetch that partial now, while this segment's MMAs
            // still run, instead of after them. Rows <= 32 only: the partial lives in registers.
            float pf[32];
            // the GEMM variants leave split tiles to w12_reduce_kernel: they only publish
            constexpr bool kFix = kArgmax;
            const bool pre_ok = kFix && !full && !dead && seg_end == r1 && c_hi - c_lo == 1 && M <= 32;
            if (pre_ok) {  // once per block: ctrl->pre is written only here
                if (et == 0) ctrl->pre = (ld_acquire_gpu(&p.tile_cnt[tile]) == 1u) ? 2 : 0;
                named_bar_sync(kEpiBar, 128);
                mode = ctrl->pre;
                if (mode == 2) {
                    fence_acq_rel_gpu();
                    const float *src = partial_of(c == c_lo ? c_hi : c_lo, tile, 0);
#pragma unroll
                    for (int i = 0; i < 32; ++i) pf[i] = (i < M) ? __ldcg(src + static_cast<size_t>(i) * kTileN) : 0.f;
                }
            }
            const bool ok = !dead && mbar_wait(smem_u32(&ctrl->accfull[b]), phb, abort, p.err, kErrEpilogue);
            // uniform over the four warps: every barrier below is taken by all of them or none
            dead = named_bar_or(kEpiBar, 128, !ok);
            const bool pre = mode == 2;  // the other block's partial is in pf
            if (!full && mode == 0) {
                if (kFix) {
                    if (et == 0)
                        ctrl->mode[par] = (ld_acquire_gpu(&p.tile_cnt[tile]) == static_cast<uint32_t>(c_hi - c_lo)) ? 2 : 1;
                    named_bar_sync(kEpiBar, 128);
                    mode = ctrl->mode[par];
                    if (mode == 2) fence_acq_rel_gpu();
                } else {
                    mode = 1;  // publish; the reduce kernel sums the tile
                }
            }
            float *part = p.partials + (static_cast<size_t>(c) * 2 + slot) * M * kTileN;
            if (!dead) {
                tc_fence_after();
                // the accumulator of each MMA issuer that had a record in this segment, added in
                // a fixed order (issuer 0, then issuer 1)
                const uint32_t lanes = static_cast<uint32_t>(32 * qw) << 16;
                const bool has0 = ((seg_start - r0) & (RPS - 1)) == 0 || seg_end - seg_start >= 2;
                const bool has1 = RPS == 2 && (((seg_start - r0) & 1) == 1 || seg_end - seg_start >= 2);
                const uint32_t t0 = tmem + lanes + (0 * p.nacc + b) * p.npad;
                const uint32_t t1 = tmem + lanes + (1 * p.nacc + b) * p.npad;
                if (pre) {
                    // two blocks: own + other is the same sum, bit for bit, in either order
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int m0 = 16 * h;
                        if (m0 >= M) break;
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
                        scale_rows(tile, f);
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] += pf[16 * h + i];
                        put_rows(m0, tile, f, nullptr);
                    }
                }
                for (int m0 = 0; !pre && m0 < M; m0 += 16) {
                    float f[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) f[i] = 0.f;
                    uint32_t v[16];
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
                    scale_rows(tile, f);
                    if (mode == 2) {
                        float acc[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            if (cc == c) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) acc[i] += f[i];
                            } else {
                                const float *src = partial_of(cc, tile, m0);
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (m0 + i < M) acc[i] += __ldcg(src + static_cast<size_t>(i) * kTileN);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] = acc[i];
                    }
                    put_rows(m0, tile, f, mode == 1 ? part : nullptr);
                }
                tc_fence_before();
            }
            mbar_arrive(smem_u32(&ctrl->accempty[b]));

            bool emitted = (mode != 1);
            if (kFix && mode == 1) {
                fence_acq_rel_gpu();  // this thread's partial stores come before the count
                named_bar_sync(kEpiBar, 128);
                if (et == 0) {
                    const uint32_t old = atomicAdd(&p.tile_cnt[tile], 1u);
                    ctrl->last[par] = (old == static_cast<uint32_t>(c_hi - c_lo)) ? 1 : 0;
                }
                named_bar_sync(kEpiBar, 128);
                emitted = ctrl->last[par] != 0;
                if (emitted) {  // published last: sum every block's partial, 16 rows at a time
                    fence_acq_rel_gpu();
                    for (int m0 = 0; m0 < M; m0 += 16) {
                        float f[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] = 0.f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            const float *src = partial_of(cc, tile, m0);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (m0 + i < M) f[i] += __ldcg(src + static_cast<size_t>(i) * kTileN);
                        }
                        put_rows(m0, tile, f, nullptr);
                    }
                }
            }
            if (mode != 0 && emitted && et == 0) p.tile_cnt[tile] = 0;  // leave the workspace zeroed
            if (kArgmax && emitted) {
                named_bar_sync(kEpiBar, 128);
                for (int m = et; m < M; m += 128) {
                    float4 a4 = ctop[m];
                    float v1 = a4.x, v2 = a4.z;
                    int i1 = __float_as_int(a4.y);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const float4 o = wtop[qq * M + m];
                        top2_merge(v1, i1, v2, o.x, __float_as_int(o.y), o.z);
                    }
                    ctop[m] = make_float4(v1, __int_as_float(i1), v2, 0.f);
                }
                named_bar_sync(kEpiBar, 128);
            }
        }
        // the tensor stores must have read their staging buffers before the block's shared
        // memory goes away (their writes to y complete on their own)
        if (!kArgmax && p.y_tma && lane == 0) bulk_wait_group_read<0>();
        if (kArgmax) {
            // publish this block's top-2 per row; the last block merges all blocks in order
            for (int m = et; m < M; m += 128) p.cta_top[static_cast<size_t>(c) * M + m] = ctop[m];
            __threadfence();
            named_bar_sync(kEpiBar, 128);
            if (et == 0) {
                const uint32_t old = atomicAdd(p.done_cnt, 1u);
                ctrl->fix = (old == static_cast<uint32_t>(G - 1)) ? 1 : 0;
            }
            named_bar_sync(kEpiBar, 128);
            if (ctrl->fix) {
                // The last block merges every block's top-2 of each row. Warp qw takes rows qw,
                // qw + 4, ...; its lanes load the blocks' top-2s 32 apart, kPer at a time with all
                // loads in flight together, and a shuffle tree merges the lanes. The top-2 of a
                // set does not depend on the merge order (equal values go to the smaller index).
                __threadfence();
                constexpr int kPer = 8;
                for (int m = qw; m < M; m += 4) {
                    float v1 = -INFINITY, v2 = -INFINITY;
                    int i1 = 0x7FFFFFFF;
                    for (int c0 = 0; c0 < G; c0 += 32 * kPer) {
                        float4 o[kPer];
#pragma unroll
                        for (int k = 0; k < kPer; ++k) {
                            const int cc = c0 + lane + 32 * k;
                            o[k] = (cc < G) ? __ldcg(p.cta_top + static_cast<size_t>(cc) * M + m)
                                            : make_float4(-INFINITY, __int_as_float(0x7FFFFFFF), -INFINITY, 0.f);
                        }
#pragma unroll
                        for (int k = 0; k < kPer; ++k) top2_merge(v1, i1, v2, o[k].x, __float_as_int(o[k].y), o[k].z);
                    }
                    warp_top2(v1, i1, v2);
                    if (lane == 0) {
                        p.idx[m] = i1;
                        p.val[m] = v1;
                        p.gap[m] = v1 - v2;
                    }
                }
                if (et == 0) *p.done_cnt = 0;
                if (et == 0 && p.run_flag) *p.run_flag = 0;  // the conditional launch has run
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (warp == kWarpProducer && lane == 0 && ctrl->abort) {
        // let copies still in flight land before the block's shared memory is released
        for (int js = (issued > S ? issued - S : 0); js < issued; ++js)  // cold path
            if (!mbar_wait_drain(smem_u32(&ctrl->full[js % S]), (js / S) & 1)) atomicOr(p.err, kErrDrain);
        for (int js = (xissued > S ? xissued - S : 0); js < xissued; ++js)
            if (!mbar_wait_drain(smem_u32(&ctrl->xfull[js % S]), (js / S) & 1)) atomicOr(p.err, kErrDrain);
    }
    if ((warp == kWarpMma || (warp == kWarpMma2 && RPS == 2)) && issued > 0) {
        const int mq = (warp == kWarpMma) ? 0 : 1;
        mma_commit_elect(smem_u32(&ctrl->done[mq]));  // same elected lane that issued the MMAs
        if (!mbar_wait_drain(smem_u32(&ctrl->done[mq]), 0) && lane == 0) atomicOr(p.err, kErrDrain);
    }
    __syncthreads();  // both issuers drained before the tensor memory is released
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split tiles of the GEMM variants (stream-K): y[m, n] = sum over the tile's blocks, in
// increasing block order, of their published fp32 partials. One block per (tile, row m), one
// thread per column of the tile; tiles covered by a single block were written by the GEMM.
// Launched right after the GEMM as a programmatic dependent launch: it waits for the GEMM's
// completion before reading the partials.
__global__ void __launch_bounds__(kTileN)
w12_reduce_kernel(const Params p) {
    grid_launch_dependents();
    const int tile = blockIdx.x, m = blockIdx.y, nl = threadIdx.x;
    const int R = p.R, G = p.grid, KT = p.k_tiles, U = p.unit, M = p.M;
    auto block_start = [&](int cc) { return U * range_start(cc, R / U, G); };
    const int c_lo = owner_of((tile * KT) / U, R / U, G);
    const int c_hi = owner_of(((tile + 1) * KT - 1) / U, R / U, G);
    if (c_lo == c_hi) return;
    grid_dependency_wait();
    const int n = tile * kTileN + nl;
    float acc = 0.f;
    constexpr int kBatch = 8;  // loads in flight per thread; the sum keeps block order
    for (int c0 = c_lo; c0 <= c_hi; c0 += kBatch) {
        float v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int cc = c0 + j;
            v[j] = 0.f;
            if (cc <= c_hi) {
                const int sl = (block_start(cc) / KT == tile) ? 0 : 1;
                v[j] = __ldcg(p.partials + ((static_cast<size_t>(cc) * 2 + sl) * M + m) * kTileN + nl);
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (c0 + j <= c_hi) acc += v[j];
    }
    if (n < p.N) {
        if (p.y_bf16)
            reinterpret_cast<__nv_bfloat16 *>(p.y)[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(acc);
        else if (p.y_accum)
            reinterpret_cast<float *>(p.y)[static_cast<size_t>(m) * p.N + n] += acc;
        else
            reinterpret_cast<float *>(p.y)[static_cast<size_t>(m) * p.N + n] = acc;
    }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

// internal operations over the INT8 head copy (reached through the certified-head entry points)
constexpr int kOpQ8 = 100;        // y = scale_n (x . q_n)
constexpr int kOpQ8Argmax = 101;  // its row argmax (the Q pass over the separate copy)
// and over the INT6 Q-pass copy (w12_q6_gemm, w12_q6_argmax)
constexpr int kOpQ6 = 102;
constexpr int kOpQ6Argmax = 103;
inline bool is_copy_op(int op) { return op == kOpQ8 || op == kOpQ8Argmax || op == kOpQ6 || op == kOpQ6Argmax; }
inline bool is_argmax_op(int op) {
    return op == W12_OP_ARGMAX || op == W12_OP_QVIEW_ARGMAX || op == kOpQ8Argmax || op == kOpQ6Argmax;
}

struct Layout {
    int npad, stages, rps, nacc, acc_cols, grid, unit, smem;
    bool whole;  // every block covers whole tiles (no partial sums)
    bool vtma;   // Q view with two records per slot: views copied through a tensor map
    bool packed; // a separate copy: INT8 (8 KB) or INT6 (6 KB) records back to back
    int64_t R;
    size_t ws_bytes, off_err, off_tile, off_done, off_part, off_top;
};

w12_status plan(const w12_tensor *t, int M, int op, Layout *L) {
    if (M < 1 || M > kMaxM) return W12_ERR_UNSUPPORTED_SHAPE;
    if ((op < W12_OP_GEMM || op > W12_OP_QVIEW_ARGMAX) && !is_copy_op(op)) return W12_ERR_INVALID_ARG;
    int sms = 0;
    W12_TRY(require_device(&sms));
    const bool q = (op == W12_OP_QVIEW_GEMM || op == W12_OP_QVIEW_ARGMAX || is_copy_op(op));
    L->packed = is_copy_op(op);
    const bool q6 = (op == kOpQ6 || op == kOpQ6Argmax);
    L->R = static_cast<int64_t>(t->n_tiles) * t->k_tiles;
    L->npad = (M + 15) / 16 * 16;
    // above 256 rows the MMA's N and the activation box are split in two halves of a multiple of 16
    if (L->npad > 256) L->npad = (M + 31) / 32 * 32;
    // two records per ring slot while the activation tiles are small
    L->rps = (L->npad <= 64) ? 2 : 1;
    // Work split. Whole tiles per block when that balances within kTileSplitSlack: no tile is
    // then shared, so no partial sums and no cross-block fix-up at the end of the launch.
    // Otherwise stream-K: equal contiguous record ranges over one block per SM.
    const int T = t->n_tiles;
    const int per = (T + sms - 1) / sms;      // tiles of the busiest block
    const int gt = (T + per - 1) / per;       // blocks needed at that load
    if (static_cast<double>(per) * sms <= kTileSplitSlack * T) {
        L->grid = gt;
        L->unit = t->k_tiles;
        L->whole = true;
    } else {
        // stream-K; small problems use fewer blocks so a tile is not split too many ways (each
        // extra block adds a partial to publish and to sum)
        const int64_t by_work = (L->R + kMinRecordsPerBlock - 1) / kMinRecordsPerBlock;
        const int64_t g = std::max<int64_t>(T, by_work);
        L->grid = static_cast<int>(std::min<int64_t>({g, L->R, static_cast<int64_t>(sms)}));
        L->unit = 1;
        L->whole = false;
    }
    // the view map needs a 16-byte aligned record array (records are 12 KB apart)
    L->vtma = q && !L->packed && L->rps == 2 && aligned16(t->records);
    const int rstride = q6 ? kQ6RecordBytes : ((L->vtma || L->packed) ? kViewBytes : kRecordBytes);
    const int rbytes = q6 ? kQ6RecordBytes : (q ? kViewBytes : kRecordBytes);
    const int sbytes = L->rps * L->npad * 128 + (L->rps - 1) * rstride + rbytes + (q ? 0 : kEscCap * 4);
    const bool am = is_argmax_op(op);
    const int ctrl = static_cast<int>(align_up(kCtrlBytes + scratch_bytes(M, am), 1024));
    int stages = (kSmemLimit - 1024 - ctrl) / sbytes;
    if (stages > kMaxStages) stages = kMaxStages;
    // tensor memory: nacc accumulators of npad columns, then 32 columns per record in flight
    // one accumulator set per MMA issuer (rps issuers), double-buffered when it fits
    // (a block of one whole tile has a single segment: nothing to double-buffer, and the
    // columns go to the ring instead)
    L->nacc = (2 * L->rps * L->npad + 4 * L->rps * kACols <= kTmemCols) ? 2 : 1;
    if (L->whole && per == 1) L->nacc = 1;
    L->acc_cols = L->rps * L->nacc * L->npad;
    const int tmem_stages = (kTmemCols - L->acc_cols) / (L->rps * kACols);
    if (stages > tmem_stages) stages = tmem_stages;
    // every decode group needs a slot of its own (the slot-ordering argument in the decode loop)
    if (stages < 2 || stages < kDecGroups) return W12_ERR_UNSUPPORTED_SHAPE;
    L->stages = stages;
    L->smem = 1024 + stages * sbytes + ctrl;
    if (L->smem < kSmemFloor) L->smem = kSmemFloor;
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

template <bool kQ, bool kA, int kPack = 0>
w12_status launch_variant(const CUtensorMap &map, const CUtensorMap &map2, const CUtensorMap &ymap,
                          const CUtensorMap &vmap, const Params &p, const Layout &L, bool overlap, cudaStream_t st) {
    auto kern = w12_gemm_kernel<kQ, kA, kPack>;
    // the opt-in shared-memory limit is set once per device (to the maximum any plan uses)
    static std::atomic<uint64_t> smem_set{0};
    int dev = 0;
    W12_CUDA(cudaGetDevice(&dev));
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!bit || !(smem_set.load(std::memory_order_acquire) & bit)) {
        W12_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit));
        smem_set.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(L.smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    W12_CUDA(cudaLaunchKernelEx(&cfg, kern, map, map2, ymap, vmap, p));
    if (!kA && !L.whole && L.grid > 1) {
        cudaLaunchConfig_t rc{};
        rc.gridDim = dim3(static_cast<unsigned>(p.n_tiles), static_cast<unsigned>(p.M));
        rc.blockDim = dim3(kTileN);
        rc.stream = st;
        rc.attrs = attr;
        rc.numAttrs = 1;  // starts while the GEMM drains; waits for it before reading
        W12_CUDA(cudaLaunchKernelEx(&rc, w12_reduce_kernel, p));
    }
    return W12_OK;
}

// ldx: elements between consecutive rows of x (K when 0)
w12_status run(const w12_tensor *t, const uint16_t *x, int M, int op, void *y, int y_dtype,
               int32_t *idx, float *val, float *gap, void *ws, size_t ws_bytes, w12_stream_t stream,
               unsigned flags = 0, const float *row_scale = nullptr, int *run_flag = nullptr, int ldx = 0) {
    if (is_copy_op(op)) {
        // a separate copy (INT8 or INT6): records and row scales only
        if (!t || !t->records || !row_scale || t->N < 1 || t->K < 1) return W12_ERR_INVALID_ARG;
    } else {
        W12_TRY(check_tensor(t));
    }
    if (flags & ~static_cast<unsigned>(W12_LAUNCH_OVERLAP | W12_LAUNCH_TEST_STALL | W12_LAUNCH_ACCUMULATE))
        return W12_ERR_INVALID_ARG;
    const bool overlap = (flags & W12_LAUNCH_OVERLAP) != 0;
    if (!x || !aligned16(x) || !ws) return W12_ERR_INVALID_ARG;
    Layout L{};
    W12_TRY(plan(t, M, op, &L));
    if (ws_bytes < L.ws_bytes) return W12_ERR_WORKSPACE;
    const bool argmax = is_argmax_op(op);
    const bool q = (op == W12_OP_QVIEW_GEMM || op == W12_OP_QVIEW_ARGMAX);
    if (argmax && (!idx || !val || !gap)) return W12_ERR_INVALID_ARG;
    if (!argmax && (!y || (y_dtype != W12_OUT_F32 && y_dtype != W12_OUT_BF16))) return W12_ERR_INVALID_ARG;
    const bool accum = (flags & W12_LAUNCH_ACCUMULATE) != 0;
    if (accum && (argmax || y_dtype != W12_OUT_F32)) return W12_ERR_INVALID_ARG;

    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return W12_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(t->K), static_cast<cuuint64_t>(M)};
    if (ldx == 0) ldx = t->K;
    if (ldx < t->K || ldx % 8 != 0) return W12_ERR_INVALID_ARG;  // rows 16-byte aligned for the copies
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
    const cuuint32_t box[2] = {kTileK, static_cast<cuuint32_t>(L.npad > 256 ? L.npad / 2 : L.npad)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return W12_ERR_INVALID_ARG;
    // x as (k within a slice, row, slice): one copy brings the slices of two consecutive records
    // as two adjacent 128B-swizzled tiles. Needs whole slices (K % 64 == 0); the single-slice
    // map above serves the other cases.
    CUtensorMap map2 = map;
    bool x_pair = false;
    if (L.rps == 2 && t->K % kTileK == 0) {
        const cuuint64_t dims3[3] = {static_cast<cuuint64_t>(kTileK), static_cast<cuuint64_t>(M),
                                     static_cast<cuuint64_t>(t->K / kTileK)};
        const cuuint64_t strides3[2] = {static_cast<cuuint64_t>(ldx) * 2, static_cast<cuuint64_t>(kTileK) * 2};
        const cuuint32_t box3[3] = {kTileK, static_cast<cuuint32_t>(L.npad), 2};
        const cuuint32_t estr3[3] = {1, 1, 1};
        x_pair = enc(&map2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(x), dims3, strides3, box3,
                     estr3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        if (!x_pair) map2 = map;
    }
    // y as a 2-D tensor for the epilogue's tiled stores (boxes of 32 columns x 16 rows); plain
    // stores are used where the tensor map's alignment rules do not hold
    CUtensorMap ymap = map;
    bool y_tma = false;
    if (!argmax) {
        const cuuint64_t esz = (y_dtype == W12_OUT_BF16) ? 2 : 4;
        const cuuint64_t ydims[2] = {static_cast<cuuint64_t>(t->N), static_cast<cuuint64_t>(M)};
        const cuuint64_t ystrides[1] = {static_cast<cuuint64_t>(t->N) * esz};
        const cuuint32_t ybox[2] = {32, 16};
        if (aligned16(y) && (ystrides[0] % 16) == 0)
            y_tma = enc(&ymap, esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y,
                        ydims, ystrides, ybox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }

    // the records as (4-byte word within a 1 KB row, row of the record, record): a box of 8 rows
    // x 2 records is two consecutive records' views, landing back to back
    CUtensorMap vmap = map;
    if (L.vtma) {
        const cuuint64_t vdims[3] = {256, kRecordBytes / 1024, static_cast<cuuint64_t>(L.R)};
        const cuuint64_t vstrides[2] = {1024, kRecordBytes};
        const cuuint32_t vbox[3] = {256, kViewBytes / 1024, 2};
        const cuuint32_t vestr[3] = {1, 1, 1};
        if (enc(&vmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, t->records, vdims, vstrides, vbox, vestr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W12_ERR_CUDA;
    }

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
    p.rps = L.rps;
    p.m3 = 8u;
    p.m15 = 32768u;
    p.nacc = L.nacc;
    p.acc_cols = L.acc_cols;
    p.grid = L.grid;
    p.unit = L.unit;
    p.overlap = overlap ? 1 : 0;
    // Tensor stores pay off when the blocks finish together (whole tiles); with split tiles
    // (stream-K) plain stores measured faster, so they are kept there.
    p.y_tma = (y_tma && L.whole) ? 1 : 0;
    p.y_accum = accum ? 1 : 0;
    p.x_pair = x_pair ? 1 : 0;
    p.v_tma = L.vtma ? 1 : 0;
    p.xhalf = (L.npad > 256) ? L.npad / 2 : 0;
    p.row_scale = row_scale;
    p.run_flag = run_flag;
    if (run_flag && (!argmax || overlap)) return W12_ERR_INVALID_ARG;  // stream-ordered argmax only
    p.test_stall = (flags & W12_LAUNCH_TEST_STALL) ? 1 : 0;
    p.R = static_cast<int>(L.R);
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
    if (op == kOpQ8) return launch_variant<true, false, 8>(map, map2, ymap, vmap, p, L, overlap, st);
    if (op == kOpQ8Argmax) return launch_variant<true, true, 8>(map, map2, ymap, vmap, p, L, overlap, st);
    if (op == kOpQ6) return launch_variant<true, false, 6>(map, map2, ymap, vmap, p, L, overlap, st);
    if (op == kOpQ6Argmax) return launch_variant<true, true, 6>(map, map2, ymap, vmap, p, L, overlap, st);
    if (q)
        return argmax ? launch_variant<true, true>(map, map2, ymap, vmap, p, L, overlap, st)
                      : launch_variant<true, false>(map, map2, ymap, vmap, p, L, overlap, st);
    return argmax ? launch_variant<false, true>(map, map2, ymap, vmap, p, L, overlap, st)
                  : launch_variant<false, false>(map, map2, ymap, vmap, p, L, overlap, st);
}

}  // namespace

// ---- entry points shared with the certified head (w12_certified.cu) ----
w12_status gemm_q8_workspace(const w12_tensor *codes, int M, size_t *bytes) {
    Layout L{};
    W12_TRY(plan(codes, M, kOpQ8, &L));
    *bytes = L.ws_bytes;
    return W12_OK;
}
w12_status gemm_q8(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, float *y, void *ws,
                   size_t ws_bytes, w12_stream_t stream) {
    return run(codes, x, M, kOpQ8, y, W12_OUT_F32, nullptr, nullptr, nullptr, ws, ws_bytes, stream, 0, row_scale);
}
w12_status gemm_q8_argmax_workspace(const w12_tensor *codes, int M, size_t *bytes) {
    Layout L{};
    W12_TRY(plan(codes, M, kOpQ8Argmax, &L));
    *bytes = L.ws_bytes;
    return W12_OK;
}
w12_status gemm_q8_argmax(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, int32_t *idx,
                          float *val, float *gap, void *ws, size_t ws_bytes, w12_stream_t stream, unsigned flags) {
    return run(codes, x, M, kOpQ8Argmax, nullptr, W12_OUT_F32, idx, val, gap, ws, ws_bytes, stream, flags,
               row_scale);
}
w12_status gemm_q6_workspace(const w12_tensor *codes, int M, bool argmax, size_t *bytes) {
    Layout L{};
    W12_TRY(plan(codes, M, argmax ? kOpQ6Argmax : kOpQ6, &L));
    *bytes = L.ws_bytes;
    return W12_OK;
}
w12_status gemm_q6(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, void *y, int y_dtype,
                   void *ws, size_t ws_bytes, w12_stream_t stream, unsigned flags) {
    return run(codes, x, M, kOpQ6, y, y_dtype, nullptr, nullptr, nullptr, ws, ws_bytes, stream, flags, row_scale);
}
w12_status gemm_q6_argmax(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, int32_t *idx,
                          float *val, float *gap, void *ws, size_t ws_bytes, w12_stream_t stream, unsigned flags) {
    return run(codes, x, M, kOpQ6Argmax, nullptr, W12_OUT_F32, idx, val, gap, ws, ws_bytes, stream, flags,
               row_scale);
}
w12_status lmhead_argmax_if(const w12_tensor *t, const uint16_t *x, int M, int32_t *idx, float *val, float *gap,
                            int *run_flag, void *ws, size_t ws_bytes, w12_stream_t stream) {
    return run(t, x, M, W12_OP_ARGMAX, nullptr, W12_OUT_F32, idx, val, gap, ws, ws_bytes, stream, 0, nullptr,
               run_flag);
}
}  // namespace w12

extern "C" w12_status w12_workspace_size(const w12_tensor *t, int M, int op, size_t *bytes) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    if (!bytes || op < W12_OP_GEMM || op > W12_OP_QVIEW_ARGMAX) return W12_ERR_INVALID_ARG;
    Layout L{};
    W12_TRY(plan(t, M, op, &L));
    *bytes = L.ws_bytes;
    return W12_OK;
}

extern "C" w12_status w12_gemm_config(const w12_tensor *t, int M, int op, int *grid, int *stages,
                                      int *smem_bytes) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    if (op < W12_OP_GEMM || op > W12_OP_QVIEW_ARGMAX) return W12_ERR_INVALID_ARG;
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

extern "C" w12_status w12_gemm_ex(const w12_tensor *t, const uint16_t *x, int M, int op, void *y,
                                  int y_dtype, int32_t *idx, float *val, float *gap, unsigned flags,
                                  void *workspace, size_t workspace_bytes, w12_stream_t stream) {
    if (op < W12_OP_GEMM || op > W12_OP_QVIEW_ARGMAX) return W12_ERR_INVALID_ARG;
    const bool argmax = (op == W12_OP_ARGMAX || op == W12_OP_QVIEW_ARGMAX);
    if (argmax && y) return W12_ERR_INVALID_ARG;
    if (!argmax && (idx || val || gap)) return W12_ERR_INVALID_ARG;
    return w12::run(t, x, M, op, y, y_dtype, idx, val, gap, workspace, workspace_bytes, stream, flags);
}

extern "C" w12_status w12_gemm_strided(const w12_tensor *t, const uint16_t *x, int ldx, int M, int op, void *y,
                                       int y_dtype, int32_t *idx, float *val, float *gap, unsigned flags,
                                       void *workspace, size_t workspace_bytes, w12_stream_t stream) {
    if (op < W12_OP_GEMM || op > W12_OP_QVIEW_ARGMAX || ldx < 1) return W12_ERR_INVALID_ARG;
    const bool argmax = (op == W12_OP_ARGMAX || op == W12_OP_QVIEW_ARGMAX);
    if (argmax && y) return W12_ERR_INVALID_ARG;
    if (!argmax && (idx || val || gap)) return W12_ERR_INVALID_ARG;
    return w12::run(t, x, M, op, y, y_dtype, idx, val, gap, workspace, workspace_bytes, stream, flags, nullptr,
                    nullptr, ldx);
}

// ------------------------------------------------------------------------------------------
// w12_gemm_noalloc: the GEMM with its workspace in a fixed device array
// ------------------------------------------------------------------------------------------
//
// Some callers cannot allocate device memory: a plug-in inside a host framework that owns all
// device memory and hands none out, or a serving loop that must not call cudaMalloc because it
// synchronises the device and can stall every stream. For them the workspace of the plain GEMM
// (the split-K counters, the error word and the fp32 partial sums of split tiles) lives in the
// file-scope array below instead. Every GPU that loads this library holds the array until the
// process exits. Its size bounds the problems this entry point accepts:
//   M <= kNoAllocMaxM rows, at most kNoAllocMaxTiles tiles of 128 output channels, and a grid of
//   at most kNoAllocMaxGrid blocks (one per SM).
constexpr int kNoAllocMaxM = 32;
constexpr int kNoAllocMaxTiles = 4096;
constexpr int kNoAllocMaxGrid = 256;
constexpr size_t kNoAllocBytes =
    256                                                          // error word
    + sizeof(uint32_t) * kNoAllocMaxTiles                        // per-tile counters
    + 256                                                        // completion counter
    + sizeof(float) * kNoAllocMaxGrid * 2 * kNoAllocMaxM * w12::kTileN  // partial sums
    + sizeof(float4) * kNoAllocMaxGrid * kNoAllocMaxM;           // per-block top-2 (argmax only)

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

namespace {
// The array's device address on the current device. In host code the symbol itself is only a
// host-side stand-in for the array, never a device address. The lookup is repeated on every
// call (it is cheap): an address cached across calls would go stale if the device's primary
// context were torn down (cudaDeviceReset) and the module loaded again elsewhere.
w12_status noalloc_scratch(void **ptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return W12_ERR_CUDA;
    *ptr = p;
    return W12_OK;
}
}  // namespace

extern "C" w12_status w12_gemm_noalloc(const w12_tensor *t, const uint16_t *x, int M, void *y,
                                       int y_dtype, w12_stream_t stream) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    if (M < 1) return W12_ERR_INVALID_ARG;
    if (M > kNoAllocMaxM || t->n_tiles > kNoAllocMaxTiles) return W12_ERR_UNSUPPORTED_SHAPE;
    Layout L{};
    W12_TRY(plan(t, M, W12_OP_GEMM, &L));
    if (L.grid > kNoAllocMaxGrid || L.ws_bytes > kNoAllocBytes) return W12_ERR_UNSUPPORTED_SHAPE;
    void *ws = nullptr;
    W12_TRY(noalloc_scratch(&ws));
    // the counters and the error word must start at zero; the partial sums need no clearing
    if (cudaMemsetAsync(ws, 0, L.off_part, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W12_ERR_CUDA;
    return run(t, x, M, W12_OP_GEMM, y, y_dtype, nullptr, nullptr, nullptr, ws, kNoAllocBytes, stream);
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
