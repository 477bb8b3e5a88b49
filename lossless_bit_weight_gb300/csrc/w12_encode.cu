// a1 — W12 encoder on the GPU.
//
// SpecPilot §4.1 "W12: A Lossless 12-bit Weight Format" and Fig. 5a: each output channel gets
// the 16-binade window [E_n-15, E_n] that holds the largest number of its weights; a weight
// whose exponent falls in it is written as three nibbles (sign and high mantissa bits, exponent
// offset, low mantissa bits), every other weight (exponent out of the window, zero, subnormal)
// is kept bit for bit in an escape list. Ties of the window choice go to the smallest E_n; placeholders, byte/nibble order and the per-record escape index follow
// the library's written format specification.
//
// Passes (all HBM-streaming, integer only):
//   window   one warp per channel: exponent histogram -> E_n, then the channel's escape count
//            per k tile (as an exclusive prefix over its k tiles, and its total) and each
//            record's total
//   scan     two blocks in one launch: exclusive prefixes over channels and over records ->
//            the offsets of both escape lists
//   pack     one block per 128x64 record: planes and escape flags of 8192 weights; the record
//            bytes, the per-record index and the per-channel list
// w12_encode_sizes runs window and scan; w12_encode reuses their results from the
// scratch and runs pack only.
#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kWindowWarps = 4;  // channels (warps) per window block (4: 56.6 us for the projection, 8: 57.9)
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 8;     // values per scan thread per tile (8: 12.0 us for the projection, 16: 14.1, 32: 13.6)
constexpr int kWinBatch = 4;    // 16-byte loads in flight per lane in the window pass
constexpr size_t kScanSmem = sizeof(uint32_t) * (kScanThreads * kScanPer + kScanThreads * kScanPer / 32);

// One warp per channel: the exponent histogram -> E_n; then the channel's escape count per k
// tile (the row read again, mostly from cache) into ct, and each count added to its record's
// total (integer atomics, so the totals do not depend on the order).
__global__ void __launch_bounds__(kWindowWarps * 32)
window_kernel(const uint16_t *__restrict__ w, int N, int K, int k_tiles, uint8_t *__restrict__ base_exp,
              uint32_t *__restrict__ ct, uint32_t *__restrict__ rec_cnt, uint32_t *__restrict__ chan_cnt) {
    __shared__ __align__(1024) uint32_t hist[kWindowWarps][256];  // 1 KB per warp, 1 KB aligned
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kWindowWarps + warp;
    uint32_t *h = hist[warp];
    for (int i = lane; i < 256; i += 32) h[i] = 0;
    __syncwarp();
    if (n < N) {
        // Both weights of a 32-bit word at once: (word >> 5) masked leaves 4 * exponent in each
        // half, OR-ed with the histogram's shared-memory address in both halves; every exponent
        // is counted (bins 0 and 255, zero/subnormal and Inf/NaN, are never read below).
        const uint32_t hb = static_cast<uint32_t>(__cvta_generic_to_shared(h));
        const uint32_t hb2 = hb | (hb << 16);  // 1 KB aligned, below 64 KB: OR adds 4 * exponent
        const uint4 *row = reinterpret_cast<const uint4 *>(w + static_cast<size_t>(n) * K);
        const int nvec = K / 8;
        // kWinBatch 16-byte loads per lane go out together, then their counts
        for (int i0 = lane; i0 < nvec; i0 += 32 * kWinBatch) {
            uint4 v[kWinBatch];
#pragma unroll
            for (int b = 0; b < kWinBatch; ++b) v[b] = (i0 + 32 * b < nvec) ? __ldg(row + i0 + 32 * b) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int b = 0; b < kWinBatch; ++b) {
                if (i0 + 32 * b >= nvec) break;
                const uint32_t wd[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t a2 = ((wd[q] >> 5) & 0x03FC03FCu) | hb2;
                    asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(a2 & 0xFFFFu) : "memory");
                    asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(a2 >> 16) : "memory");
                }
            }
        }
    }
    __syncwarp();
    // best window: largest coverage, then smallest base. Lane l holds bins 8l .. 8l + 7 as the
    // histogram's inclusive prefix P; the window [E - 15, E] covers P[E] - P[E - 16] weights,
    // P[E - 16] being the same slot of lane l - 2
    uint32_t P[8];
    {
        const uint4 h0 = reinterpret_cast<const uint4 *>(h)[2 * lane];
        const uint4 h1 = reinterpret_cast<const uint4 *>(h)[2 * lane + 1];
        P[0] = h0.x; P[1] = h0.y; P[2] = h0.z; P[3] = h0.w;
        P[4] = h1.x; P[5] = h1.y; P[6] = h1.z; P[7] = h1.w;
    }
#pragma unroll
    for (int j = 1; j < 8; ++j) P[j] += P[j - 1];
    uint32_t incl = P[7];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    const uint32_t lane_before = incl - P[7];
    uint32_t best_c = 0;
    int best_E = 1 << 30;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        P[j] += lane_before;
        const uint32_t lo = __shfl_up_sync(0xFFFFFFFFu, P[j], 2);
        const int E = 8 * lane + j;
        const uint32_t c = P[j] - lo;
        if (E >= 16 && E <= 254 && (c > best_c || (c == best_c && E < best_E))) {
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
    const uint32_t lo2 = static_cast<uint32_t>(best_E - 15) * 0x00010001u;
    const uint4 *row = reinterpret_cast<const uint4 *>(w + static_cast<size_t>(n) * K);
    const int nvec = K / 8;
    const int nt = n / kTileN;
    // kWinBatch chunks of 32 pieces (4 k tiles each) per round of loads; the counts become this
    // channel's exclusive prefix over its k tiles (ct) and its total (chan_cnt) on the way
    uint32_t run = 0;  // escapes of this channel in earlier k tiles
    for (int j00 = 0; j00 < 8 * k_tiles; j00 += 32 * kWinBatch) {
        uint4 v[kWinBatch];
#pragma unroll
        for (int b = 0; b < kWinBatch; ++b) {
            const int i = j00 + 32 * b + lane;
            v[b] = (n < N && i < nvec) ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int b = 0; b < kWinBatch; ++b) {
            const int j0 = j00 + 32 * b;
            if (j0 >= 8 * k_tiles) break;
            const int i = j0 + lane;
            uint32_t c = 0;
            if (n < N && i < nvec) {
                // two weights per word: D = E - lo_e + 256 per half (no borrow between halves);
                // outside the window iff bits 4..8 of D differ from 10000b; the flags land in
                // bits 9 and 25 and are summed as two 16-bit fields
                const uint32_t wd[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
                uint32_t acc = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t D = ((wd[q] >> 7) & 0x00FF00FFu) + 0x01000100u - lo2;
                    acc += (((D ^ 0x01000100u) & 0x01F001F0u) + 0x01F001F0u) & 0x02000200u;
                }
                c = ((acc >> 9) & 0xFFFFu) + (acc >> 25);
            }
            c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
            c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
            c += __shfl_xor_sync(0xFFFFFFFFu, c, 4);
            // the chunk's four k-tile counts (octets 0..3) and this octet's prefix among them
            const uint32_t c0 = __shfl_sync(0xFFFFFFFFu, c, 0), c1 = __shfl_sync(0xFFFFFFFFu, c, 8);
            const uint32_t c2 = __shfl_sync(0xFFFFFFFFu, c, 16), c3 = __shfl_sync(0xFFFFFFFFu, c, 24);
            const int oct = lane >> 3;
            const uint32_t before = run + (oct > 0 ? c0 : 0u) + (oct > 1 ? c1 : 0u) + (oct > 2 ? c2 : 0u);
            const int kt = i >> 3;
            if ((lane & 7) == 0 && kt < k_tiles) {
                ct[static_cast<size_t>(n) * k_tiles + kt] = before;
                if (c) atomicAdd(&rec_cnt[static_cast<size_t>(nt) * k_tiles + kt], c);
            }
            run += c0 + c1 + c2 + c3;
        }
    }
    if (lane == 0) chan_cnt[n] = run;
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
// its share of the per-channel lists; at most 40 registers, so that six blocks share an SM
__global__ void __launch_bounds__(256, 6) pack_kernel(PackArgs a) {
    const int r = blockIdx.x;
    const int nt = r / a.k_tiles, kt = r % a.k_tiles;
    const int nl = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int n = nt * kTileN + nl;
    const int k0 = kt * kTileK + 32 * half;
    const int En = a.base_exp[n];
    // the offsets this thread needs after the block scan, requested now so their latency
    // overlaps the weight loads and the encoding
    const uint32_t rec_off_r = a.rec_off[r];
    const uint32_t chan_off_n = (n < a.N) ? a.chan_off[n] : 0u;
    const uint32_t ct_nk = (n < a.N) ? a.ct[static_cast<size_t>(n) * a.k_tiles + kt] : 0u;

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

    // Planes of a weight under the window [lo_e, lo_e + 15] = [E_n - 15, E_n] (format rules 2
    // and 3): inside it, view byte = (E - lo_e) << 4 | m_hi << 1 | s and B = the low mantissa
    // nibble. Two weights per 32-bit word at a time (weight 2p in the low half of u[p], 2p + 1
    // in the high half), every weight first encoded as if inside the window; the escapes, rare,
    // get their placeholder codes below. Per half: D = E - lo_e + 256 lies in [2, 510] (no
    // borrow between the halves), the weight is inside iff D >> 4 == 16, and then its exponent
    // code is D & 15.
    const uint32_t lo2 = static_cast<uint32_t>(En - 15) * 0x00010001u;
    uint32_t view16[16], lo16[16];
    uint32_t mask = 0;  // escape flags, bit j <-> k0 + j
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const uint32_t w2 = u[q];
        const uint32_t D = ((w2 >> 7) & 0x00FF00FFu) + 0x01000100u - lo2;
        const uint32_t viol = (D ^ 0x01000100u) & 0x01F001F0u;  // nonzero in a half iff outside
        view16[q] = ((D & 0x000F000Fu) << 4) | ((w2 >> 3) & 0x000E000Eu) | ((w2 >> 15) & 0x00010001u);
        lo16[q] = w2 & 0x000F000Fu;
        const uint32_t e2 = (viol + 0x01F001F0u) & 0x02000200u;  // bit 9: weight 2q, bit 25: 2q + 1
        mask |= ((e2 >> 9) & 1u) << (2 * q);
        mask |= (e2 >> 25) << (2 * q + 1);
    }
    uint32_t vw[8], bw[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) vw[i] = __byte_perm(view16[2 * i], view16[2 * i + 1], 0x6420);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        bw[i] = lo16[4 * i] | (lo16[4 * i + 1] << 4) | (lo16[4 * i + 2] << 8) | (lo16[4 * i + 3] << 12);
    // weights past the matrix (rows n >= N, columns k >= K: whole groups of 8) hold zero codes
    const int vk = (n < a.N) ? min(32, max(0, a.K - k0)) : 0;
    if (vk < 32) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (4 * i >= vk) vw[i] = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (8 * i >= vk) bw[i] = 0;
        mask &= (vk > 0) ? (0xFFFFFFFFu >> (32 - vk)) : 0u;
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
    const int64_t seg = static_cast<int64_t>(rec_off_r);
    if (total > 0 && (threadIdx.x & 63) == 63) {  // last thread of 32-row quarter q
        const int64_t hi = seg + (threadIdx.x >> 6);
        if (hi < a.rec_cap) a.rec_esc[hi] = rank + cnt;
    }
    const int64_t rbase = seg + 4 + rank;
    // canonical per-channel list: this channel's escapes in earlier k tiles come first
    const int64_t cbase = (n < a.N) ? static_cast<int64_t>(chan_off_n) + ct_nk + (half ? partner : 0) : 0;
    // Escapes are rare (about one per record): their patterns are read again (from L2) rather
    // than kept live across the block scan. Each one's record bytes, written above with the
    // in-window codes, get their placeholders here: the view byte (above the window E = 15,
    // m_hi = 7; below it zero; the sign stays), and the plane-B byte it shares with weight j ^ 2
    // (B = 15 above the window, 0 below, the weight's own low bits inside).
    const uint16_t *wrow = a.w + static_cast<size_t>(n) * a.K + k0;
    auto low_code = [&](uint32_t b) -> uint32_t {
        const int e = static_cast<int>((b >> 7) & 0xFFu);
        return (e > En) ? 0xFu : ((e < En - 15) ? 0u : (b & 0xFu));
    };
    uint32_t seen = 0;
    for (uint32_t m = mask; m != 0; m &= m - 1) {
        const int j = __ffs(m) - 1;
        const uint32_t bits = __ldg(wrow + j);
        const uint32_t bits2 = __ldg(wrow + (j ^ 2));
        const bool above = static_cast<int>((bits >> 7) & 0xFFu) > En;
        rec[2048 * (2 * half + (j >> 4)) + 16 * nl + (j & 15)] = static_cast<uint8_t>((above ? 0xFEu : 0u) | (bits >> 15));
        const int i8 = j & 7, nib = (i8 >> 1) + 4 * (i8 & 1);
        const uint32_t lj = low_code(bits), lp = low_code(bits2);
        rec[kViewBytes + 2048 * half + 16 * nl + 4 * (j >> 3) + (nib >> 1)] =
            static_cast<uint8_t>((nib & 1) ? (lp | (lj << 4)) : (lj | (lp << 4)));
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

// Block b runs job b (the channel scan and the record scan share one launch). The input goes
// through shared memory a tile of kScanThreads * kScanPer values at a time: read and written
// back with coalesced accesses, each thread summing and then prefixing its own kScanPer
// consecutive values there, with a block scan of the thread sums in between and the running
// total carried from tile to tile.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanJob j0, ScanJob j1) {
    const ScanJob &job = blockIdx.x == 0 ? j0 : j1;
    const uint32_t *in = job.in;
    const int64_t count = job.count;
    uint32_t *out = job.out;
    const int seg = job.seg;
    extern __shared__ uint32_t tile[];  // kScanThreads * kScanPer (+ 1 per 32, against bank conflicts)
    __shared__ uint32_t warp_sums[kScanThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    auto at = [](int i) { return i + (i >> 5); };  // padded index: a thread's kScanPer values span banks
    uint32_t carry = 0;
    constexpr int kTile = kScanThreads * kScanPer;
    for (int64_t base = 0; base < count; base += kTile) {
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
            const int i = j * kScanThreads + t;
            const uint32_t v = (base + i < count) ? in[base + i] : 0u;
            tile[at(i)] = seg ? segment_words(v) : v;
        }
        __syncthreads();
        uint32_t local = 0;
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) local += tile[at(t * kScanPer + j)];
        uint32_t incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {  // inclusive scan of the 32 warp sums
            uint32_t x = warp_sums[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, x, off);
                if (lane >= off) x += o;
            }
            warp_sums[lane] = x;
        }
        __syncthreads();
        const uint32_t before = warp ? warp_sums[warp - 1] : 0u, all = warp_sums[kScanThreads / 32 - 1];
        uint32_t run = carry + before + incl - local;
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
            const uint32_t v = tile[at(t * kScanPer + j)];
            tile[at(t * kScanPer + j)] = run;
            run += v;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
            const int i = j * kScanThreads + t;
            if (base + i < count) out[base + i] = tile[at(i)];
        }
        carry += all;
        __syncthreads();  // the tile and warp_sums are reused
    }
    if (t == 0) out[count] = carry;
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
    window_kernel<<<n_pad / kWindowWarps, kWindowWarps * 32, 0, st>>>(w, N, K, k_tiles, base_exp, s.ct, s.rec_cnt,
                                                                       s.chan_cnt);
    W12_CUDA(cudaGetLastError());
    static const cudaError_t scan_attr =
        cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kScanSmem));
    W12_CUDA(scan_attr);
    scan_kernel<<<2, kScanThreads, kScanSmem, st>>>(ScanJob{s.chan_cnt, N, esc_off, 0}, ScanJob{s.rec_cnt, R, rec_off, 1});
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
