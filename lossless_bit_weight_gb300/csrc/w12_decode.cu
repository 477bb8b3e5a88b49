// a2 — W12 decode and the load-time bit-for-bit check.
//
// SpecPilot §4.1 and the caption of Table A2: when the model loads, each decoded tensor is
// compared bit for bit with the checkpoint. One block per 128x64 record: 256 threads, each
// decodes 32 weights of one channel row (two view chunks, one plane-B chunk) with the same
// in-register decode the GEMM uses, then the record's escapes are restored from the per-record
// index. HBM-bound: 1.5 B/weight read (+2 B/weight written or compared).
#include "w12_internal.cuh"

namespace w12 {
namespace {

// decode the 32 weights k_l = 32*half .. 32*half+31 of row n_l of a record in global memory
__device__ __forceinline__ void decode_half_row(const uint8_t *rec, int nl, int half, int En,
                                                uint32_t (&out)[16]) {
    const uint4 v0 = __ldg(reinterpret_cast<const uint4 *>(rec + 2048 * (2 * half) + 16 * nl));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4 *>(rec + 2048 * (2 * half + 1) + 16 * nl));
    const uint4 b = __ldg(reinterpret_cast<const uint4 *>(rec + kViewBytes + 2048 * half + 16 * nl));
    const uint32_t base2 = base2_of(En);
    decode_chunk16<false, 0>(v0, b, base2, out);
    decode_chunk16<false, 1>(v1, b, base2, out + 8);
}

__global__ void __launch_bounds__(256)
decode_kernel(const uint8_t *__restrict__ records, const uint8_t *__restrict__ base_exp,
              const uint32_t *__restrict__ rec_off, const uint32_t *__restrict__ rec_esc, int N,
              int K, int k_tiles, uint16_t *__restrict__ w_out) {
    const int r = blockIdx.x;
    const int nt = r / k_tiles, kt = r % k_tiles;
    const int nl = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int n = nt * kTileN + nl;
    const int k0 = kt * kTileK + 32 * half;
    const uint8_t *rec = records + static_cast<size_t>(r) * kRecordBytes;
    uint32_t out[16];
    decode_half_row(rec, nl, half, base_exp[n], out);
    if (n < N) {
        uint16_t *dst = w_out + static_cast<size_t>(n) * K + k0;
#pragma unroll
        for (int g = 0; g < 4; ++g)
            if (k0 + 8 * g < K)
                reinterpret_cast<uint4 *>(dst)[g] =
                    make_uint4(out[4 * g], out[4 * g + 1], out[4 * g + 2], out[4 * g + 3]);
    }
    __syncthreads();  // escapes overwrite placeholders written above by other threads
    // a non-empty segment starts with a 4-word header of quarter ends
    const uint32_t first = rec_off[r] + (rec_off[r + 1] > rec_off[r] ? 4u : 0u);
    for (uint32_t i = first + threadIdx.x; i < rec_off[r + 1]; i += blockDim.x) {
        const uint32_t e = rec_esc[i];
        const uint32_t pos = e & 0xFFFFu;
        if (pos >= static_cast<uint32_t>(kRecordWeights)) continue;  // padding entry
        const int en = nt * kTileN + static_cast<int>(pos >> 6);
        const int ek = kt * kTileK + static_cast<int>(pos & 63u);
        if (en < N && ek < K) w_out[static_cast<size_t>(en) * K + ek] = static_cast<uint16_t>(e >> 16);
    }
}

// counters[0] += differing weights/entries, counters[1] += real per-record index entries.
// The record's planes and the reference row chunks are loaded first: they do not depend on the
// escape pass, so their latency overlaps it. Two block barriers; counts are summed per warp.
__global__ void __launch_bounds__(256)
verify_kernel(const uint8_t *__restrict__ records, const uint8_t *__restrict__ base_exp,
              const uint32_t *__restrict__ rec_off, const uint32_t *__restrict__ rec_esc, int N,
              int K, int k_tiles, const uint16_t *__restrict__ w_ref,
              unsigned long long *counters) {
    __shared__ uint32_t esc_map[kRecordWeights / 32];
    __shared__ uint32_t quarter_cnt[4];
    const int r = blockIdx.x;
    const int nt = r / k_tiles, kt = r % k_tiles;
    const int nl = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int n = nt * kTileN + nl;
    const int k0 = kt * kTileK + 32 * half;
    const uint8_t *rec = records + static_cast<size_t>(r) * kRecordBytes;
    const uint4 v0 = __ldg(reinterpret_cast<const uint4 *>(rec + 2048 * (2 * half) + 16 * nl));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4 *>(rec + 2048 * (2 * half + 1) + 16 * nl));
    const uint4 bq = __ldg(reinterpret_cast<const uint4 *>(rec + kViewBytes + 2048 * half + 16 * nl));
    const int En = base_exp[n];
    uint4 ref[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
        ref[g] = (n < N && k0 + 8 * g < K)
                     ? __ldg(reinterpret_cast<const uint4 *>(w_ref + static_cast<size_t>(n) * K + k0 + 8 * g))
                     : make_uint4(0, 0, 0, 0);
    const uint32_t seg_lo = rec_off[r], seg_hi = rec_off[r + 1];

    esc_map[threadIdx.x] = 0;  // 256 words, one per thread
    if (threadIdx.x < 4) quarter_cnt[threadIdx.x] = 0;
    __syncthreads();
    uint32_t bad = 0, entries = 0;
    const uint32_t first = seg_lo + (seg_hi > seg_lo ? 4u : 0u);
    for (uint32_t i = first + threadIdx.x; i < seg_hi; i += blockDim.x) {
        const uint32_t e = rec_esc[i];
        if (e == 0xFFFFFFFFu) continue;  // padding entry
        const uint32_t pos = e & 0xFFFFu;
        const int en = nt * kTileN + static_cast<int>(pos >> 6);
        const int ek = kt * kTileK + static_cast<int>(pos & 63u);
        if (pos >= static_cast<uint32_t>(kRecordWeights) || en >= N || ek >= K) {
            ++bad;
            continue;
        }
        ++entries;
        atomicAdd(&quarter_cnt[pos >> 11], 1u);
        atomicOr(&esc_map[pos >> 5], 1u << (pos & 31u));
        if (static_cast<uint16_t>(e >> 16) != w_ref[static_cast<size_t>(en) * K + ek]) ++bad;
    }
    __syncthreads();
    // the header the GEMM reads must hold the cumulative quarter counts
    if (threadIdx.x == 0 && seg_hi > seg_lo) {
        uint32_t run = 0;
        for (int q = 0; q < 4; ++q) {
            run += quarter_cnt[q];
            if (rec_esc[seg_lo + q] != run) ++bad;
        }
    }
    uint32_t out[16];
    const uint32_t base2 = base2_of(En);
    decode_chunk16<false, 0>(v0, bq, base2, out);
    decode_chunk16<false, 1>(v1, bq, base2, out + 8);
    if (n < N) {
        const uint32_t emask = esc_map[(nl * kTileK + 32 * half) >> 5];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (k0 + 8 * g >= K) continue;
            const uint32_t rw[4] = {ref[g].x, ref[g].y, ref[g].z, ref[g].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t diff = out[4 * g + q] ^ rw[q];
                const int j = 8 * g + 2 * q;
                if (!((emask >> j) & 1u) && (diff & 0xFFFFu)) ++bad;
                if (!((emask >> (j + 1)) & 1u) && (diff >> 16)) ++bad;
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        bad += __shfl_xor_sync(0xFFFFFFFFu, bad, off);
        entries += __shfl_xor_sync(0xFFFFFFFFu, entries, off);
    }
    if ((threadIdx.x & 31) == 0) {
        if (bad) atomicAdd(&counters[0], static_cast<unsigned long long>(bad));
        if (entries) atomicAdd(&counters[1], static_cast<unsigned long long>(entries));
    }
}

// canonical list: each entry must name an in-range k, in increasing order, with the exact bits
__global__ void verify_csr_kernel(const uint32_t *__restrict__ esc_off,
                                  const uint32_t *__restrict__ esc_k,
                                  const uint16_t *__restrict__ esc_bits, int N, int K,
                                  const uint16_t *__restrict__ w_ref, unsigned long long *counters) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    uint32_t bad = 0;
    int64_t prev = -1;
    for (uint32_t i = esc_off[n]; i < esc_off[n + 1]; ++i) {
        const uint32_t k = esc_k[i];
        if (static_cast<int64_t>(k) <= prev || k >= static_cast<uint32_t>(K)) {
            ++bad;
            continue;
        }
        prev = k;
        if (esc_bits[i] != w_ref[static_cast<size_t>(n) * K + k]) ++bad;
    }
    if (bad) atomicAdd(&counters[2], static_cast<unsigned long long>(bad));
}

}  // namespace
}  // namespace w12

extern "C" w12_status w12_decode(const w12_tensor *t, uint16_t *w_out, w12_stream_t stream) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    if (!w_out || !aligned16(w_out)) return W12_ERR_INVALID_ARG;
    W12_TRY(require_device(nullptr));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int R = t->n_tiles * t->k_tiles;
    decode_kernel<<<R, 256, 0, st>>>(t->records, t->base_exp, t->rec_esc_off, t->rec_esc, t->N,
                                     t->K, t->k_tiles, w_out);
    W12_CUDA(cudaGetLastError());
    return W12_OK;
}

extern "C" w12_status w12_verify_scratch_size(size_t *bytes) {
    if (!bytes) return W12_ERR_INVALID_ARG;
    *bytes = 4 * sizeof(unsigned long long);
    return W12_OK;
}

extern "C" w12_status w12_verify(const w12_tensor *t, const uint16_t *w_ref, void *scratch,
                                 size_t scratch_bytes, uint64_t *n_mismatch, w12_stream_t stream) {
    using namespace w12;
    W12_TRY(check_tensor(t));
    if (!w_ref || !aligned16(w_ref) || !scratch || !n_mismatch) return W12_ERR_INVALID_ARG;
    if (scratch_bytes < 4 * sizeof(unsigned long long)) return W12_ERR_WORKSPACE;
    W12_TRY(require_device(nullptr));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long *cnt = static_cast<unsigned long long *>(scratch);
    W12_CUDA(cudaMemsetAsync(cnt, 0, 4 * sizeof(unsigned long long), st));
    const int R = t->n_tiles * t->k_tiles;
    verify_kernel<<<R, 256, 0, st>>>(t->records, t->base_exp, t->rec_esc_off, t->rec_esc, t->N,
                                     t->K, t->k_tiles, w_ref, cnt);
    W12_CUDA(cudaGetLastError());
    if (t->n_esc > 0) {
        verify_csr_kernel<<<static_cast<int>(ceil_div(t->N, 256)), 256, 0, st>>>(
            t->esc_off, t->esc_k, t->esc_bits, t->N, t->K, w_ref, cnt);
        W12_CUDA(cudaGetLastError());
    }
    unsigned long long h[4] = {0, 0, 0, 0};
    uint32_t csr_total = 0;
    W12_CUDA(cudaMemcpyAsync(h, cnt, sizeof h, cudaMemcpyDeviceToHost, st));
    W12_CUDA(cudaMemcpyAsync(&csr_total, t->esc_off + t->N, 4, cudaMemcpyDeviceToHost, st));
    W12_CUDA(cudaStreamSynchronize(st));
    uint64_t bad = h[0] + h[2];
    // both lists must describe the same number of escapes as the tensor header
    const int64_t rec_entries = static_cast<int64_t>(h[1]);
    bad += static_cast<uint64_t>(rec_entries > t->n_esc ? rec_entries - t->n_esc : t->n_esc - rec_entries);
    const int64_t csr = csr_total;
    bad += static_cast<uint64_t>(csr > t->n_esc ? csr - t->n_esc : t->n_esc - csr);
    *n_mismatch = bad;
    return bad ? W12_ERR_MISMATCH : W12_OK;
}
