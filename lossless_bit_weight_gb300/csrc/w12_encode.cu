// a1 — W12 encoder on the GPU.
//
// SpecPilot §4.1 "W12: A Lossless 12-bit Weight Format" and Fig. 5a: per output channel choose
// the 16-binade window [E_n-15, E_n] covering the most weights; store in-window weights as a
// sign/top-mantissa nibble, an exponent-offset nibble and a low-mantissa nibble; send weights
// outside the window, zeros and denormals to an exact escape list. Ties of the window choice
// go to the smallest E_n; placeholders, byte/nibble order and the per-record escape index follow
// the library's written format specification.
//
// Passes (all HBM-streaming, integer only):
//   window   one warp per channel: exponent histogram -> E_n, then the channel's escape count
//            per k tile and each record's total
//   rowscan  one warp per channel: exclusive prefix of its per-k-tile counts
//   scan     two blocks in one launch: exclusive prefixes over channels and over records ->
//            the offsets of both escape lists
//   pack     one block per 128x64 record: planes and escape flags of 8192 weights; the record
//            bytes, the per-record index and the per-channel list
// w12_encode_sizes runs window, rowscan and scan; w12_encode reuses their results from the
// scratch and runs pack only.
#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kWindowWarps = 8;
constexpr int kScanThreads = 1024;

// planes of a real weight u under the window [lo_e, lo_e + 15] = [E_n - 15, E_n] (format rules 2
// and 3), without branches. E_n lies in [16, 254], so the window holds normal exponents only: a
// weight is inside iff its biased exponent lies in it, above it (larger, Inf, NaN: clamped to the
// window top, E = 15, m_hi = 7, B = 15) or below it (smaller, zero, subnormal: E = m_hi = B = 0).
__device__ __forceinline__ void planes(uint32_t u, int lo_e, uint32_t &view, uint32_t &lo, bool &esc) {
    const int x = static_cast<int>((u >> 7) & 0xFFu) - lo_e;  // exponent offset in the window
    const bool inside = static_cast<uint32_t>(x) <= 15u;
    const uint32_t t = inside ? (u & 0x7Fu) : (x > 15 ? 0x7Fu : 0u);  // mantissa or its clamp
    const uint32_t dc = static_cast<uint32_t>(min(max(x, 0), 15));
    view = (dc << 4) | ((t >> 3) & 0xEu) | (u >> 15);
    lo = t & 0xFu;
    esc = !inside;
}

// One warp per channel: the exponent histogram -> E_n; then the channel's escape count per k
// tile (the row read again, mostly from cache) into ct, and each count added to its record's
// total (integer atomics, so the totals do not depend on the order).
__global__ void __launch_bounds__(kWindowWarps * 32)
window_kernel(const uint16_t *__restrict__ w, int N, int K, int k_tiles, uint8_t *__restrict__ base_exp,
              uint32_t *__restrict__ ct, uint32_t *__restrict__ rec_cnt) {
    __shared__ uint32_t hist[kWindowWarps][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kWindowWarps + warp;
    uint32_t *h = hist[warp];
    for (int i = lane; i < 256; i += 32) h[i] = 0;
    __syncwarp();
    if (n < N) {
        const uint4 *row = reinterpret_cast<const uint4 *>(w + static_cast<size_t>(n) * K);
        const int nvec = K / 8;
        for (int i = lane; i < nvec; i += 32) {
            const uint4 v = __ldg(row + i);
            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t u = (wd[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
                const uint32_t e = (u >> 7) & 0xFFu;
                if (e >= 1u && e <= 254u) atomicAdd(&h[e], 1u);
            }
        }
    }
    __syncwarp();
    // best window: largest coverage, then smallest base
    uint32_t best_c = 0;
    int best_E = 1 << 30;
    for (int E = 16 + lane; E <= 254; E += 32) {
        uint32_t c = 0;
#pragma unroll
        for (int d = 0; d < 16; ++d) c += h[E - d];
        if (c > best_c || (c == best_c && E < best_E)) {
            best_c = c;
            best_E = E;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const uint32_t oc = __shfl_xor_sync(0xFFFFFFFFu, best_c, off);
        const int oE = __shfl_xor_sync(0xFFFFFFFFu, best_E, off);
        if (oc > best_c || (oc == best_c && oE < best_E)) {
            best_c = oc;
            best_E = oE;
        }
    }
    if (lane == 0) base_exp[n] = static_cast<uint8_t>(n < N ? best_E : 16);
    // escapes per k tile: lane l holds 16-byte piece i = l + 32 j (k = 8 i .. 8 i + 7), so the 8
    // lanes of each lane octet share one k tile (4 j + l / 8); a weight stays in the window iff
    // its biased exponent lies in [E_n - 15, E_n] (that range holds normal exponents only)
    const uint32_t lo_e = static_cast<uint32_t>(best_E - 15);
    const uint4 *row = reinterpret_cast<const uint4 *>(w + static_cast<size_t>(n) * K);
    const int nvec = K / 8;
    const int nt = n / kTileN;
    for (int j0 = 0; j0 < 8 * k_tiles; j0 += 32) {
        const int i = j0 + lane;
        uint32_t c = 0;
        if (n < N && i < nvec) {
            const uint4 v = __ldg(row + i);
            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t e = (wd[q >> 1] >> (16 * (q & 1) + 7)) & 0xFFu;
                c += (e - lo_e > 15u) ? 1u : 0u;
            }
        }
        c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
        c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
        c += __shfl_xor_sync(0xFFFFFFFFu, c, 4);
        const int kt = i >> 3;
        if ((lane & 7) == 0 && kt < k_tiles) {
            ct[static_cast<size_t>(n) * k_tiles + kt] = c;
            if (c) atomicAdd(&rec_cnt[static_cast<size_t>(nt) * k_tiles + kt], c);
        }
    }
}

struct PackArgs {
    const uint16_t *w;
    int N, K, k_tiles;
    const uint8_t *base_exp;
    const uint32_t *ct;  // [n_pad * k_tiles] per-(channel, k-tile) exclusive prefixes
    uint8_t *records;
    const uint32_t *rec_off;
    uint32_t *rec_esc;
    int64_t rec_cap;
    const uint32_t *chan_off;
    uint32_t *esc_k;
    uint16_t *esc_bits;
    int64_t esc_cap;
};

// exclusive prefix of `v` over the 256 threads of the block (thread order); *total = block sum
__device__ __forceinline__ uint32_t block_excl_scan256(uint32_t v, uint32_t *total) {
    __shared__ uint32_t warp_sums[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t s = warp_sums[i];
        if (i < warp) before += s;
        all += s;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

// one block per record: planes of its 128 x 64 weights, the record bytes, its index segment and
// its share of the per-channel lists
__global__ void __launch_bounds__(256) pack_kernel(PackArgs a) {
    const int r = blockIdx.x;
    const int nt = r / a.k_tiles, kt = r % a.k_tiles;
    const int nl = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int n = nt * kTileN + nl;
    const int k0 = kt * kTileK + 32 * half;
    const int En = a.base_exp[n];

    uint32_t u[16];  // 32 bf16 patterns, two per word, k ascending
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n < a.N && k0 + 8 * g < a.K)
            v = __ldg(reinterpret_cast<const uint4 *>(a.w + static_cast<size_t>(n) * a.K + k0 + 8 * g));
        u[4 * g + 0] = v.x;
        u[4 * g + 1] = v.y;
        u[4 * g + 2] = v.z;
        u[4 * g + 3] = v.w;
    }

    uint32_t vw[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // view bytes, 4 per word
    uint32_t bw[4] = {0, 0, 0, 0};              // B nibbles, 8 per word
    uint32_t mask = 0;                          // escape flags, bit j <-> k0 + j
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t bits = (u[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
        const bool real = (n < a.N) && (k0 + j < a.K);
        uint32_t view = 0, lo = 0;
        bool esc = false;
        if (real) planes(bits, En - 15, view, lo, esc);
        vw[j >> 2] |= view << (8 * (j & 3));
        const int i = j & 7;
        bw[j >> 3] |= lo << (4 * ((i >> 1) + 4 * (i & 1)));
        if (esc) mask |= 1u << j;
    }
    const uint32_t cnt = __popc(mask);
    const uint32_t partner = __shfl_xor_sync(0xFFFFFFFFu, cnt, 1);

    uint8_t *rec = a.records + static_cast<size_t>(r) * kRecordBytes;
    reinterpret_cast<uint4 *>(rec + 2048 * (2 * half) + 16 * nl)[0] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
    reinterpret_cast<uint4 *>(rec + 2048 * (2 * half + 1) + 16 * nl)[0] = make_uint4(vw[4], vw[5], vw[6], vw[7]);
    reinterpret_cast<uint4 *>(rec + kViewBytes + 2048 * half + 16 * nl)[0] = make_uint4(bw[0], bw[1], bw[2], bw[3]);

    // per-record index: a 4-word header of quarter ends, then the entries in increasing
    // pos = 64*n_l + k_l (thread order), then padding to a multiple of 4 words
    uint32_t total;
    const uint32_t rank = block_excl_scan256(cnt, &total);
    const int64_t seg = static_cast<int64_t>(a.rec_off[r]);
    if (total > 0 && (threadIdx.x & 63) == 63) {  // last thread of 32-row quarter q
        const int64_t hi = seg + (threadIdx.x >> 6);
        if (hi < a.rec_cap) a.rec_esc[hi] = rank + cnt;
    }
    const int64_t rbase = seg + 4 + rank;
    // canonical per-channel list: this channel's escapes in earlier k tiles come first
    const int64_t cbase = (n < a.N) ? static_cast<int64_t>(a.chan_off[n]) +
                                          a.ct[static_cast<size_t>(n) * a.k_tiles + kt] +
                                          (half ? partner : 0)
                                    : 0;
    // escapes are rare (about one per record): their patterns are read again (from L2) rather
    // than keeping the 32 loaded patterns live across the block scan, which cost occupancy
    uint32_t seen = 0;
    for (uint32_t m = mask; m != 0; m &= m - 1) {
        const int j = __ffs(m) - 1;
        const uint32_t bits = __ldg(a.w + static_cast<size_t>(n) * a.K + k0 + j);
        const int64_t ri = rbase + seen, ci = cbase + seen;
        if (ri < a.rec_cap)
            a.rec_esc[ri] = static_cast<uint32_t>(nl * kTileK + 32 * half + j) | (bits << 16);
        if (ci < a.esc_cap) {
            a.esc_k[ci] = static_cast<uint32_t>(k0 + j);
            a.esc_bits[ci] = static_cast<uint16_t>(bits);
        }
        ++seen;
    }
    if (threadIdx.x == 255 && total > 0) {
        const int64_t end = a.rec_off[r + 1];
        for (int64_t i = seg + 4 + total; i < end; ++i)
            if (i < a.rec_cap) a.rec_esc[i] = 0xFFFFFFFFu;
    }
}

// one warp per channel: exclusive prefix of its per-k-tile counts, in place, and the total
__global__ void __launch_bounds__(256) rowscan_kernel(uint32_t *ct, int n_pad, int k_tiles, uint32_t *chan_cnt) {
    const int n = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (n >= n_pad) return;
    uint32_t *row = ct + static_cast<size_t>(n) * k_tiles;
    uint32_t run = 0;
    for (int k0 = 0; k0 < k_tiles; k0 += 32) {
        const int kt = k0 + lane;
        const uint32_t c = (kt < k_tiles) ? row[kt] : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += o;
        }
        if (kt < k_tiles) row[kt] = run + incl - c;
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) chan_cnt[n] = run;
}

// words of a record's index segment with c escapes: none, or a 4-word header + c entries
// rounded up to a multiple of 4
__device__ __forceinline__ uint32_t segment_words(uint32_t c) { return c ? 4u + ((c + 3u) & ~3u) : 0u; }

// out[i] = sum_{j<i} in'[j], out[count] = total, with in' = in, or segment_words(in) if seg
struct ScanJob {
    const uint32_t *in;
    int64_t count;
    uint32_t *out;
    int seg;
};

// block b runs job b (the channel scan and the record scan share one launch)
__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanJob j0, ScanJob j1) {
    const ScanJob &job = blockIdx.x == 0 ? j0 : j1;
    const uint32_t *in = job.in;
    const int64_t count = job.count;
    uint32_t *out = job.out;
    const int seg = job.seg;
    __shared__ uint32_t warp_sums[kScanThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t chunk = (count + kScanThreads - 1) / kScanThreads;
    const int64_t lo = t * chunk, hi = (lo + chunk < count) ? lo + chunk : count;
    uint32_t local = 0;
    for (int64_t i = lo; i < hi; ++i) {
        const uint32_t v = in[i];
        local += seg ? segment_words(v) : v;
    }
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
    for (int i = 0; i < kScanThreads / 32; ++i) {
        if (i < warp) before += warp_sums[i];
        all += warp_sums[i];
    }
    uint32_t run = before + incl - local;
    for (int64_t i = lo; i < hi; ++i) {
        const uint32_t v = in[i];
        out[i] = run;
        run += seg ? segment_words(v) : v;
    }
    if (t == 0) out[count] = all;
}

struct Scratch {
    uint8_t *base_tmp;
    uint32_t *ct, *rec_cnt, *chan_cnt, *off_chan, *off_rec;
    size_t bytes;
};

Scratch carve(void *base, int N, int K) {
    const int64_t n_pad = ceil_div(N, kTileN) * kTileN;
    const int64_t k_tiles = ceil_div(K, kTileK);
    const int64_t R = (n_pad / kTileN) * k_tiles;
    Scratch s{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_base = take(n_pad);
    const size_t o_ct = take(sizeof(uint32_t) * n_pad * k_tiles);
    const size_t o_rc = take(sizeof(uint32_t) * R);
    const size_t o_cc = take(sizeof(uint32_t) * n_pad);
    const size_t o_oc = take(sizeof(uint32_t) * (N + 1));
    const size_t o_or = take(sizeof(uint32_t) * (R + 1));
    s.bytes = off;
    uint8_t *b = static_cast<uint8_t *>(base);
    if (b) {
        s.base_tmp = b + o_base;
        s.ct = reinterpret_cast<uint32_t *>(b + o_ct);
        s.rec_cnt = reinterpret_cast<uint32_t *>(b + o_rc);
        s.chan_cnt = reinterpret_cast<uint32_t *>(b + o_cc);
        s.off_chan = reinterpret_cast<uint32_t *>(b + o_oc);
        s.off_rec = reinterpret_cast<uint32_t *>(b + o_or);
    }
    return s;
}

// window + counting passes + offsets; base_exp, esc_off, rec_off may point at scratch
w12_status count_pass(const uint16_t *w, int N, int K, const Scratch &s, uint8_t *base_exp,
                      uint32_t *esc_off, uint32_t *rec_off, cudaStream_t st) {
    const int n_tiles = static_cast<int>(ceil_div(N, kTileN));
    const int k_tiles = static_cast<int>(ceil_div(K, kTileK));
    const int n_pad = n_tiles * kTileN;
    const int R = n_tiles * k_tiles;
    W12_CUDA(cudaMemsetAsync(s.rec_cnt, 0, sizeof(uint32_t) * static_cast<size_t>(R), st));
    window_kernel<<<n_pad / kWindowWarps, kWindowWarps * 32, 0, st>>>(w, N, K, k_tiles, base_exp, s.ct, s.rec_cnt);
    W12_CUDA(cudaGetLastError());
    rowscan_kernel<<<static_cast<int>(ceil_div(n_pad, 8)), 256, 0, st>>>(s.ct, n_pad, k_tiles, s.chan_cnt);
    W12_CUDA(cudaGetLastError());
    scan_kernel<<<2, kScanThreads, 0, st>>>(ScanJob{s.chan_cnt, N, esc_off, 0}, ScanJob{s.rec_cnt, R, rec_off, 1});
    W12_CUDA(cudaGetLastError());
    return W12_OK;
}

}  // namespace
}  // namespace w12

extern "C" w12_status w12_encode_scratch_size(int N, int K, size_t *bytes) {
    using namespace w12;
    if (!bytes) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(N, K));
    *bytes = carve(nullptr, N, K).bytes;
    return W12_OK;
}

extern "C" w12_status w12_encode_sizes(const uint16_t *w, int N, int K, void *scratch,
                                       size_t scratch_bytes, int64_t *n_esc, int64_t *n_rec_esc,
                                       w12_stream_t stream) {
    using namespace w12;
    if (!w || !scratch || !n_esc || !n_rec_esc) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(N, K));
    if (!aligned16(w) || !aligned16(scratch)) return W12_ERR_INVALID_ARG;
    W12_TRY(require_device(nullptr));
    const Scratch s = carve(scratch, N, K);
    if (scratch_bytes < s.bytes) return W12_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    W12_TRY(count_pass(w, N, K, s, s.base_tmp, s.off_chan, s.off_rec, st));
    const int64_t R = ceil_div(N, kTileN) * ceil_div(K, kTileK);
    uint32_t tot[2] = {0, 0};
    W12_CUDA(cudaMemcpyAsync(&tot[0], s.off_chan + N, 4, cudaMemcpyDeviceToHost, st));
    W12_CUDA(cudaMemcpyAsync(&tot[1], s.off_rec + R, 4, cudaMemcpyDeviceToHost, st));
    W12_CUDA(cudaStreamSynchronize(st));
    *n_esc = tot[0];
    *n_rec_esc = tot[1];
    return W12_OK;
}

extern "C" w12_status w12_encode(const uint16_t *w, int N, int K, void *scratch,
                                 size_t scratch_bytes, const w12_tensor *t, w12_stream_t stream) {
    using namespace w12;
    if (!w || !scratch || !t) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(N, K));
    W12_TRY(check_tensor(t));
    if (t->N != N || t->K != K) return W12_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(scratch)) return W12_ERR_INVALID_ARG;
    W12_TRY(require_device(nullptr));
    const Scratch s = carve(scratch, N, K);
    if (scratch_bytes < s.bytes) return W12_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int R = t->n_tiles * t->k_tiles;
    // the window bases, per-(channel, k tile) prefixes and both offset lists are those that
    // w12_encode_sizes left in the scratch for this w: copy the three outputs into place
    const size_t n_pad = static_cast<size_t>(t->n_tiles) * kTileN;
    W12_CUDA(cudaMemcpyAsync(t->base_exp, s.base_tmp, n_pad, cudaMemcpyDeviceToDevice, st));
    W12_CUDA(cudaMemcpyAsync(t->esc_off, s.off_chan, sizeof(uint32_t) * (static_cast<size_t>(N) + 1),
                             cudaMemcpyDeviceToDevice, st));
    W12_CUDA(cudaMemcpyAsync(t->rec_esc_off, s.off_rec, sizeof(uint32_t) * (static_cast<size_t>(R) + 1),
                             cudaMemcpyDeviceToDevice, st));
    PackArgs a{};
    a.w = w;
    a.N = N;
    a.K = K;
    a.k_tiles = t->k_tiles;
    a.base_exp = t->base_exp;
    a.ct = s.ct;
    a.records = t->records;
    a.rec_off = t->rec_esc_off;
    a.rec_esc = t->rec_esc;
    a.rec_cap = t->n_rec_esc;
    a.chan_off = t->esc_off;
    a.esc_k = t->esc_k;
    a.esc_bits = t->esc_bits;
    a.esc_cap = t->n_esc;
    pack_kernel<<<R, 256, 0, st>>>(a);
    W12_CUDA(cudaGetLastError());
    uint32_t tot[2] = {0, 0};
    W12_CUDA(cudaMemcpyAsync(&tot[0], t->esc_off + N, 4, cudaMemcpyDeviceToHost, st));
    W12_CUDA(cudaMemcpyAsync(&tot[1], t->rec_esc_off + R, 4, cudaMemcpyDeviceToHost, st));
    W12_CUDA(cudaStreamSynchronize(st));
    if (tot[0] != t->n_esc || tot[1] != t->n_rec_esc) return W12_ERR_INVALID_ARG;
    return W12_OK;
}
