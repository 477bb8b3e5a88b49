// Internal helpers of the W12 CUDA library (sm_103a only): status plumbing, inline-PTX wrappers
// for mbarriers, bulk/tensor copies and the tcgen05 tensor-core instructions, bounded waits.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w12.h"

namespace w12 {

constexpr int kTileN = 128;
constexpr int kTileK = 64;
constexpr int kRecordBytes = 12288;
constexpr int kViewBytes = 8192;
constexpr int kRecordWeights = kTileN * kTileK;  // 8192
constexpr int kQ6RecordBytes = W12_Q6_RECORD_BYTES;  // 6144: the INT6 copy's record

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

#define W12_TRY(expr)                         \
    do {                                      \
        w12_status _st = (expr);              \
        if (_st != W12_OK) return _st;        \
    } while (0)

#define W12_CUDA(expr)                                  \
    do {                                                \
        cudaError_t _e = (expr);                        \
        if (_e != cudaSuccess) return W12_ERR_CUDA;     \
    } while (0)

// The current device must be a compute capability 10.3 GPU; checked once per device.
w12_status require_device(int *sm_count);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

w12_status check_shape(int N, int K);
// cuTensorMapEncodeTiled from the driver, or null if the driver does not provide it
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
w12_status check_tensor(const w12_tensor *t);

// GEMM entry points shared between translation units (defined in w12_gemm.cu):
// the GEMM over the certified head's INT8 copy (records in `codes->records`, 8 KB each; y fp32)
w12_status gemm_q8_workspace(const w12_tensor *codes, int M, size_t *bytes);
w12_status gemm_q8(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, float *y, void *ws,
                   size_t ws_bytes, w12_stream_t stream);
// the row argmax over the INT8 copy (flags: W12_LAUNCH_OVERLAP)
w12_status gemm_q8_argmax_workspace(const w12_tensor *codes, int M, size_t *bytes);
w12_status gemm_q8_argmax(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, int32_t *idx,
                          float *val, float *gap, void *ws, size_t ws_bytes, w12_stream_t stream, unsigned flags);
// the GEMM and the row argmax over the INT6 Q-pass copy (6 KB records; flags: W12_LAUNCH_OVERLAP)
w12_status gemm_q6_workspace(const w12_tensor *codes, int M, bool argmax, size_t *bytes);
w12_status gemm_q6(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, void *y, int y_dtype,
                   void *ws, size_t ws_bytes, w12_stream_t stream, unsigned flags);
w12_status gemm_q6_argmax(const w12_tensor *codes, const float *row_scale, const uint16_t *x, int M, int32_t *idx,
                          float *val, float *gap, void *ws, size_t ws_bytes, w12_stream_t stream, unsigned flags);
// the W12 head's fused argmax, launched stream-ordered; it does nothing unless *run_flag != 0
// when it starts, and clears the flag when it has run
w12_status lmhead_argmax_if(const w12_tensor *t, const uint16_t *x, int M, int32_t *idx, float *val, float *gap,
                            int *run_flag, void *ws, size_t ws_bytes, w12_stream_t stream);

// ------------------------------------------------------------------------------------------
// device side
// ------------------------------------------------------------------------------------------

// error bits written to the workspace error word by a kernel that gives up a wait
enum : int {
    kErrProducer = 1,
    kErrEscape = 2,
    kErrDecode = 4,
    kErrMma = 8,
    kErrEpilogue = 16,
    kErrDrain = 32,
};

// bounded waits give up after this long (ns of %globaltimer)
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;
constexpr uint64_t kDrainLimitNs = 100ull * 1000ull * 1000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Non-blocking probe of a phase (no suspension; the fast path of a wait that is already done).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Blocking probe: the thread sleeps (issuing nothing) until the phase completes or about
// `kSuspendNs` pass, so waiting warps leave the issue slots to the working ones.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete. Gives up (returns false) when
// another role of the block has raised `abort`, or after kWaitLimitNs; in the latter case it
// raises `abort` and records `code` in the global error word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *gerr, int code) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 3u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(gerr, code);
                return false;
            }
        }
    }
}

// Short wait used only while draining on the way out of a kernel.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kDrainLimitNs) return false;
    }
    return true;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0, both 16B aligned)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 2-D tiled tensor copy global -> shared (box and swizzle from the tensor map)
__device__ __forceinline__ void tma_2d_g2s(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 2-D tiled tensor copy shared -> global (bulk async-group of the executing thread); elements
// of the box outside the tensor are not written
__device__ __forceinline__ void tma_2d_s2g(const CUtensorMap *map, int c0, int c1, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
        ::"l"(map), "r"(c0), "r"(c1), "r"(src)
        : "memory");
}
// the same box added element-wise into global memory (y += staged values; one addition each)
__device__ __forceinline__ void tma_2d_s2g_add(const CUtensorMap *map, int c0, int c1, uint32_t src) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];"
        ::"l"(map), "r"(c0), "r"(c1), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk groups still have to read their shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// order this thread's generic-proxy shared-memory writes before later async-proxy reads
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch (sm_90+). wait: block until the grids this launch depends on
// have completed and their memory is visible (returns at once when there are none).
// launch_dependents: let the grid launched after this one on the stream begin; it still waits
// for this grid's completion before reading anything this grid produced.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---- issue from a converged warp -------------------------------------------------------------
// The copy-engine and tensor-core instructions below are issued once per warp by the lane that
// elect.sync picks (the same lane every time when the whole warp is active), with the rest of the
// warp converged and computing the same operands. Issuing them from a single diverged thread
// costs several times more cycles per instruction on sm_103.

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
        "@P mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}"
        ::"r"(bar), "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
        "@P mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}"
        ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_elect(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
        "@P cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_3d_g2s_elect(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                                 uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
        "@P cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n\t}"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_2d_g2s_elect(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
        "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n\t}"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, tensor memory) ---------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 with bf16 inputs and fp32 accumulation, M = 128.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA issued by the elected lane of a converged warp.
__device__ __forceinline__ void mma_bf16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                  uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred P;\n\t.reg .pred A;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "setp.ne.b32 A, %4, 0;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, A;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same, always accumulating into D (no predicate to compute).
__device__ __forceinline__ void mma_bf16_ts_acc_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                      uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred P;\n\t.reg .pred A;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "setp.eq.u32 A, 1, 1;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, A;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc)
        : "memory");
}

// Four MMAs of one 128 x 64 record and the commit that tracks them, from one elected lane:
// A = 32 tensor-memory columns from a_tmem (8 per K = 16 step), B = the 128B-swizzled activation
// tile of b_desc (32 bytes, 2 in the descriptor's address field, per step). The first MMA
// overwrites D unless `accumulate`.
__device__ __forceinline__ void mma4_bf16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred P;\n\t.reg .pred A;\n\t.reg .pred T;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "setp.ne.b32 A, %4, 0;\n\t"
        "setp.eq.u32 T, 1, 1;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, A;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, T;\n\t"
        "@P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate),
          "r"(a_tmem + 8), "l"(b_desc + 2), "r"(a_tmem + 16), "l"(b_desc + 4), "r"(a_tmem + 24), "l"(b_desc + 6),
          "r"(bar)
        : "memory");
}

// The same for more than 256 activation rows: the MMA's N is split into two halves of nh rows
// (nh <= 256, a multiple of 16): per K step one MMA into accumulator columns [0, nh) from the
// tile's first nh rows and one into [nh, 2 nh) from the next nh rows (b_desc + b_half), then
// one commit for all eight.
__device__ __forceinline__ void mma4x2_bf16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                     uint64_t b_half, uint32_t nh, uint32_t idesc,
                                                     uint32_t accumulate, uint32_t bar) {
    const uint32_t d1 = d_tmem + nh;
    const uint64_t c = b_desc + b_half;
    asm volatile(
        "{\n\t.reg .pred P;\n\t.reg .pred A;\n\t.reg .pred T;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "setp.ne.b32 A, %5, 0;\n\t"
        "setp.eq.u32 T, 1, 1;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %3, %6, A;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %4, %6, A;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %6, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%1], [%7], %9, %6, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%10], %11, %6, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%1], [%10], %12, %6, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%0], [%13], %14, %6, T;\n\t"
        "@P tcgen05.mma.cta_group::1.kind::f16 [%1], [%13], %15, %6, T;\n\t"
        "@P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%16];\n\t}"
        ::"r"(d_tmem), "r"(d1), "r"(a_tmem), "l"(b_desc), "l"(c), "r"(accumulate), "r"(idesc),
          "r"(a_tmem + 8), "l"(b_desc + 2), "l"(c + 2), "r"(a_tmem + 16), "l"(b_desc + 4), "l"(c + 4),
          "r"(a_tmem + 24), "l"(b_desc + 6), "l"(c + 6), "r"(bar)
        : "memory");
}

// Commit from the elected lane (the lane that issued the MMAs it must track).
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\t"
        "@P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Each lane stores 32 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// One 32-bit column of the warp's 32 lanes (each lane its own value).
__device__ __forceinline__ uint32_t tmem_ld_32x32b_x1(uint32_t taddr) {
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr) : "memory");
    return v;
}
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Each lane loads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the 128-byte swizzle
// (rows of 64 bf16 = 128 B, 8-row atoms 1024 B apart), as a TMA SWIZZLE_128B box lays it out.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);        // start address
    d |= static_cast<uint64_t>(1u) << 16;                       // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;               // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1u) << 46;                       // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                       // swizzle: 128B
    return d;
}

// Instruction descriptor for kind::f16: bf16 A and B (K-major), fp32 D, shape 128 x n.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t m, uint32_t n) {
    return (1u << 4)              // D format: f32
         | (1u << 7)              // A format: bf16
         | (1u << 10)             // B format: bf16
         | ((n >> 3) << 17)       // N / 8
         | ((m >> 4) << 24);      // M / 16
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A release increment of a counter (gpu scope): the writes that happen before it in this block
// (the calling thread's, and the other threads' before a block barrier that the caller passed) are
// visible to a thread that reads the incremented value with an acquire load.
__device__ __forceinline__ void red_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The same with the old value returned and acquire semantics as well: the caller (and, after a
// block barrier, its block) sees every write released by the increments before this one.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// named barrier that also ORs a predicate over the participating threads
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// ---- in-register W12 decode -------------------------------------------------------------
//
// Two weights (k = 2p, 2p+1) become one bf16x2 word, low half = even k.
//   x     = view bytes of the two weights at bits 0..7 and 16..23 (byte = E<<4 | m_hi<<1 | s)
//   bs    = plane-B word shifted so the two low-mantissa nibbles sit at bits 0..3 and 16..19
//   base2 = (E_n - 15) << 7 in both halves
//   m3 = 8, m15 = 32768 (the multipliers of the two shifts)
// t = x*8 + base2 puts m_hi at bits 4..6 and E + E_n - 15 (<= 254: no carry into the sign) at
// bits 7..14; its stray sign bit lands at bit 3, which the nibble select overwrites.
// u = x*32768 puts each sign at bit 15 / 31. Callers that are bound by the integer ALU pass
// the multipliers as run-time values so both run as multiply-adds on the FMA pipe; the ALU
// then does one byte permute and two 3-input logic ops per word.
template <bool kQView>
__device__ __forceinline__ uint32_t decode_pair(uint32_t x, uint32_t bs, uint32_t base2, uint32_t m3,
                                                uint32_t m15) {
    // Written as PTX so that each bit-field select stays one lop3 (select LUT 0xCA: a ? b : c);
    // from the C++ form the compiler emitted two logic ops for one of them.
    uint32_t t, u, r1, out;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(t) : "r"(x), "r"(m3), "r"(base2));
    asm("mul.lo.u32 %0, %1, %2;" : "=r"(u) : "r"(x), "r"(m15));
    asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(r1) : "r"(0x80008000u), "r"(u), "r"(t));  // sign | rest
    if (kQView) {  // low mantissa := 1000b: (r1 & 0xFFF0FFF0) | 0x00080008 (LUT 0xEA)
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(out) : "r"(r1), "r"(0xFFF0FFF0u), "r"(0x00080008u));
        return out;
    }
    asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(out) : "r"(0x000F000Fu), "r"(bs), "r"(r1));  // B nibbles
    return out;
}

// Sixteen weights k_l = 16c .. 16c+15 of one channel row -> 8 bf16x2 words.
//   v = the row's 16 view bytes of chunk c; b = the row's 16 plane-B bytes of chunk c >> 1;
//   kOdd = c & 1 (selects which half of the plane-B chunk holds these k).
template <bool kQView, int kOdd>
__device__ __forceinline__ void decode_chunk16(const uint4 &v, const uint4 &b, uint32_t base2,
                                               uint32_t *out, uint32_t m3 = 8u,
                                               uint32_t m15 = 32768u) {
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t B = bw[2 * kOdd + (q >> 1)];
        const int sh = 8 * (q & 1);
        out[2 * q] = decode_pair<kQView>(__byte_perm(vw[q], 0u, 0x4140u), B >> sh, base2, m3, m15);
        out[2 * q + 1] = decode_pair<kQView>(__byte_perm(vw[q], 0u, 0x4342u), B >> (sh + 4), base2, m3, m15);
    }
}

// Two sign-magnitude INT8 codes (bit 7 sign, bits 0-6 magnitude m; the certified head's copy)
// -> one bf16x2 word of their integer values, exactly. A byte permute places code i in the low
// byte of half i with its sign replicated through the high byte; then h = sign | 0x4300 | m is
// +-(128 + m) and c = sign | 0x4300 is +-128, and h - c = +-m exactly.
__device__ __forceinline__ uint32_t decode_q8_pair(uint32_t codes, uint32_t sel) {
    uint32_t x, h, c, out;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(codes), "r"(sel));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(h) : "r"(x), "r"(0x807F807Fu), "r"(0x43004300u));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(c) : "r"(x), "r"(0x80008000u), "r"(0x43004300u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(h), "r"(c));
    return out;
}

// Sixteen INT8 codes k_l = 16c .. 16c+15 of one row -> 8 bf16x2 words.
__device__ __forceinline__ void decode_q8_chunk16(const uint4 &v, uint32_t *out) {
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        out[2 * q] = decode_q8_pair(vw[q], 0x9180u);      // codes 0, 1 of the word
        out[2 * q + 1] = decode_q8_pair(vw[q], 0xB3A2u);  // codes 2, 3
    }
}

// Sixteen INT6 codes k_l = 16g .. 16g+15 of one row -> 8 bf16x2 words (word j: k_l = 16g + 2j
// in the low half, 16g + 2j + 1 in the high half). Each code c is stored as u = c + 32 (1..63):
// lw0 / lw1 are the row's plane-L words 2g and 2g+1 (the low four bits of pair j at bits 4(j&3)
// and 16 + 4(j&3) of word j >> 2), tw its plane-T word g (the top two bits of pair j at bits 2j
// and 16 + 2j). OR-ing u into the mantissa of 128.0 (bf16 0x4300, whose mantissa step is 1)
// gives 128 + u exactly, and subtracting 160 leaves c exactly.
__device__ __forceinline__ void decode_q6_group16(uint32_t lw0, uint32_t lw1, uint32_t tw, uint32_t *out) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t l = ((j < 4) ? lw0 : lw1) >> (4 * (j & 3));
        const uint32_t t = (j < 2) ? (tw << (4 - 2 * j)) : (tw >> (2 * j - 4));  // bits 2j -> 4
        uint32_t v, o;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(l), "r"(0x000F000Fu), "r"(0x43004300u));
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(t), "r"(0x00300030u), "r"(v));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(o) : "r"(v), "r"(0x43204320u));
        out[j] = o;
    }
}

// ---- arithmetic of the layer stream's row normalisation (shared by its kernels) ----------

// bf16 bits of a double, rounded to nearest even in one step: on the bit pattern for results in
// the normal range (the 52-bit mantissa rounded to 7 bits; a carry moves into the exponent, and
// an exponent beyond 127 gives Inf), by an exact scaling to the subnormal quantum 2^-133 below.
__device__ __forceinline__ uint16_t bf16_bits_rne(double v) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(v));
    const uint16_t sign = static_cast<uint16_t>((b >> 48) & 0x8000u);
    const uint64_t a = b & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return 0x7FC0;  // NaN
    if (a < 0x3810000000000000ull)  // below 2^-126: the bf16 subnormal range; 128 = smallest normal
        return sign | static_cast<uint16_t>(rint(__longlong_as_double(static_cast<long long>(a)) * 0x1p133));
    const uint64_t r = (a + 0x0FFFFFFFFFFFull + ((a >> 45) & 1u)) >> 45;  // exponent field | 7 mantissa bits
    const int e = static_cast<int>(r >> 7) - 1023 + 127;
    if (e >= 255) return sign | 0x7F80;
    return sign | static_cast<uint16_t>((e << 7) | static_cast<int>(r & 0x7Fu));
}

// v * 2^s exactly (up to the final rounding of a subnormal result, as ldexpf): one multiply when
// 2^s is a normal fp32 value
__device__ __forceinline__ float scale_pow2(float v, int s) {
    if (s >= -126 && s <= 127) return __fmul_rn(v, __uint_as_float(static_cast<uint32_t>(127 + s) << 23));
    return ldexpf(v, s);
}

// The two rare cases of bf16_mul_rne below, kept out of line so the common path stays short.
static __device__ __noinline__ uint16_t bf16_mul_rne_f64(float w, float yh, float yl) {
    return bf16_bits_rne(static_cast<double>(w) * (static_cast<double>(yh) + static_cast<double>(yl)));
}
static __device__ __noinline__ uint16_t bf16_mul_rne_mid(float w, float yh, float yl, float p) {
    const uint32_t bits = __float_as_uint(p);
    const float m = __uint_as_float((bits & 0xFFFF0000u) | 0x8000u);
    const float t = __fadd_rn(__fmaf_rn(w, yh, -p), __fmul_rn(w, yl));
    float d = __fadd_rn(__fsub_rn(p, m), t);  // w y - m, its sign exact but for a cancellation below 2^-149
    if (bits >> 31) d = -d;                   // in magnitude
    const uint32_t down = bits >> 16;         // the neighbour toward zero
    if (d > 0.f) return static_cast<uint16_t>(down + 1u);
    if (d < 0.f) return static_cast<uint16_t>(down);
    return static_cast<uint16_t>(down + (down & 1u));  // on the midpoint: the even neighbour
}

// bf16 bits of w * y, nearest even, for y = yh + yl (|yl| <= ulp(yh) / 2) and w fp32, without fp64
// in the common case. p = fl(w yh) is within 1.5 fp32 ulps of w y (the product's rounding error
// plus w yl), so unless p lies within one ulp of the midpoint between its two bf16 neighbours,
// p rounds like w y. Near the midpoint m, the sign of (p - m) + (w yh - p) + w yl decides (p - m
// is exact; the product error comes from an FMA). Results near or below the fp32 normal range,
// and non-finite ones, take the fp64 route.
__device__ __forceinline__ uint16_t bf16_mul_rne(float w, float yh, float yl) {
    const float p = __fmul_rn(w, yh);
    const uint32_t bits = __float_as_uint(p);
    const uint32_t mag = bits & 0x7FFFFFFFu;
    if (mag < 0x04000000u || mag >= 0x7F000000u) return bf16_mul_rne_f64(w, yh, yl);  // |p| < 2^-119, >= 2^127
    if ((bits & 0xFFFFu) - 0x7FFFu <= 2u) return bf16_mul_rne_mid(w, yh, yl, p);     // within an ulp of the midpoint
    return static_cast<uint16_t>((bits + 0x7FFFu + ((bits >> 16) & 1u)) >> 16);
}

struct F2 {  // an unevaluated sum hi + lo of two fp32 values
    float hi, lo;
};
// a double as an fp32 pair hi + lo (host or device)
__host__ __device__ inline F2 f2_of(double v) {
    const float hi = static_cast<float>(v);
    return {hi, static_cast<float>(v - static_cast<double>(hi))};
}
// a + b, with the rounding error of the leading addition carried into lo (two-sum)
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    const float s = __fadd_rn(a.hi, b.hi);
    const float bb = __fsub_rn(s, a.hi);
    const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
    const float lo = __fadd_rn(__fadd_rn(a.lo, b.lo), err);
    const float hi = __fadd_rn(s, lo);  // renormalise (|s| >= |lo|)
    return {hi, __fsub_rn(lo, __fsub_rn(hi, s))};
}

// 1 / rms of a row from the sum t (fp32 pair) of the squares of its values scaled by 2^-e and 1/K as
// an fp32 pair: the fp32 reciprocal square root y0 of the mean and one Newton step,
// y1 = y0 + y0 (1 - mean y0^2) / 2, with the residual formed in fp32 pairs (the square of y0 and
// the products exact through FMAs; 1 - q is exact since q is within a few ulps of 1), about 2^-43
// relative; returned as an fp32 pair. The row's x = bf16(h / rms(h)) is then
// bf16_mul_rne(h * 2^-e, yh, yl).
struct RmsScale {
    float yh, yl;
};
__device__ __forceinline__ RmsScale rms_scale(F2 t, F2 inv_k) {
    // mean = t * inv_k as a pair (mh, ml)
    const float p = __fmul_rn(t.hi, inv_k.hi);
    float pe = __fmaf_rn(t.hi, inv_k.hi, -p);
    pe = __fadd_rn(pe, __fadd_rn(__fmul_rn(t.hi, inv_k.lo), __fmul_rn(t.lo, inv_k.hi)));
    const float mh = __fadd_rn(p, pe);
    const float ml = __fsub_rn(pe, __fsub_rn(mh, p));
    const float y0 = rsqrtf(mh);
    // mean * y0^2 = q + qe
    const float s = __fmul_rn(y0, y0);
    const float se = __fmaf_rn(y0, y0, -s);
    const float q = __fmul_rn(mh, s);
    float qe = __fmaf_rn(mh, s, -q);
    qe = __fadd_rn(qe, __fadd_rn(__fmul_rn(mh, se), __fmul_rn(ml, s)));
    const float r = __fsub_rn(__fsub_rn(1.f, q), qe);
    const float corr = __fmul_rn(__fmul_rn(0.5f, y0), r);
    const float yh = __fadd_rn(y0, corr);
    return {yh, __fsub_rn(corr, __fsub_rn(yh, y0))};
}

__device__ __forceinline__ uint32_t base2_of(int En) {
    const uint32_t b = static_cast<uint32_t>(En - 15) << 7;
    return b | (b << 16);
}

}  // namespace w12
