// us_encode.cu -- dense -> bitmap tiles on the GPU.
//
// Format: IE-BME of "UnionSparse: An Index-Efficient Sparsity Framework for
// Low-Bit Sparse LLM Inference on Edge", section V-A (Union Bitmaps, Union
// Value Offsets o_t = sum of earlier payload lengths, Compressed Values
// CV[o_t + rho]) with one area (Q = 1), scanned row-major or column-major
// (Tiled-CBC, "Unified Static-Dynamic Pruning for Efficient LLM Inference"
// section 4.1), each tile's run padded to 16 bytes (same page, 4.2.3).
//
// Three launches:
//   1. count: one CTA per tile builds the tile's 64-bit words and stores P_t
//      (its popcount);
//   2. scan:  one CTA turns roundup(P_t, E) into the exclusive prefix tile_off;
//   3. pack:  one CTA per tile ranks its set positions (word prefix +
//      masked popcount), compacts them in shared memory and writes the run,
//      zero padding included, with 16-byte stores.
// Row-scan tiles 64 columns wide (a row of the tile is one bitmap word) whose
// rows start on 16-byte boundaries take count and pack kernels that read W
// 16 bytes per lane: the nonzero bytes / halves of a load become mask bits by
// word-parallel bit tricks, and the lanes of one row combine their pieces of
// the row word by shuffles.  Every other shape takes kernels that read W one
// element per lane, with warp ballots over the scan positions.
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kEncThreads = 256;

template <int ELEM>
__device__ __forceinline__ bool is_nonzero(const void* W, int64_t idx) {
    if (ELEM == US_F16) return (reinterpret_cast<const uint16_t*>(W)[idx] & 0x7FFFu) != 0;
    return reinterpret_cast<const int8_t*>(W)[idx] != 0;
}

// position p of a TM x TK tile -> offset (i*ldw + j) from the tile's corner
__device__ __forceinline__ int64_t pos_offset(int order, int TM, int TK, int p, int64_t ldw) {
    int i, j;
    if (order == US_ORDER_ROW) { i = p / TK; j = p - i * TK; }
    else                       { j = p / TM; i = p - j * TM; }
    return (int64_t)i * ldw + j;
}

template <int ELEM>
__global__ void __launch_bounds__(kEncThreads)
enc_count_kernel(const void* __restrict__ W, int64_t ldw, int TM, int TK, int nTK, int order,
                 uint64_t* __restrict__ bitmap, uint32_t* __restrict__ counts, unsigned* status) {
    const int t = blockIdx.x;
    const int tm = t / nTK, tk = t - tm * nTK;
    const int64_t corner = (int64_t)tm * TM * ldw + (int64_t)tk * TK;
    const int nw = TM * TK / 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int warp_sum[kEncThreads / 32];
    int my = 0;
    for (int w = warp; w < nw; w += kEncThreads / 32) {
        const int p0 = w * 64 + lane, p1 = p0 + 32;
        const int64_t i0 = corner + pos_offset(order, TM, TK, p0, ldw);
        const int64_t i1 = corner + pos_offset(order, TM, TK, p1, ldw);
        const bool nz0 = is_nonzero<ELEM>(W, i0), nz1 = is_nonzero<ELEM>(W, i1);
        if (ELEM != US_F16) {
            const int lo = ELEM == US_I4 ? -8 : -2, hi = ELEM == US_I4 ? 7 : 1;
            const int8_t a = reinterpret_cast<const int8_t*>(W)[i0];
            const int8_t b = reinterpret_cast<const int8_t*>(W)[i1];
            if (a < lo || a > hi || b < lo || b > hi) us::set_status(status, US_ERR_INVALID_ARG);
        }
        const uint32_t lo = __ballot_sync(0xffffffffu, nz0);
        const uint32_t hi = __ballot_sync(0xffffffffu, nz1);
        if (lane == 0) {
            bitmap[(int64_t)t * nw + w] = (uint64_t)lo | ((uint64_t)hi << 32);
            my += __popc(lo) + __popc(hi);
        }
    }
    if (lane == 0) warp_sum[warp] = my;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int i = 0; i < kEncThreads / 32; ++i) s += warp_sum[i];
        counts[t] = (uint32_t)s;
    }
}

// Exclusive scan of the padded run lengths; one CTA of 1024 threads, four
// tiles a thread per pass (counts is 16-byte aligned, passes start at
// multiples of 4096 tiles), so a 4096-tile matrix takes one pass.
__global__ void __launch_bounds__(1024)
enc_scan_kernel(const uint32_t* __restrict__ counts, int64_t nT, int E, uint32_t* __restrict__ tile_off,
                unsigned* status) {
    __shared__ uint32_t wsum[32];
    __shared__ uint64_t carry_s;
    if (threadIdx.x == 0) { carry_s = 0; tile_off[0] = 0; }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t base = 0; base < nT; base += 4096) {
        const int64_t t0 = base + 4 * (int64_t)threadIdx.x;
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (t0 + 3 < nT) {
            const uint4 c = *reinterpret_cast<const uint4*>(counts + t0);
            v[0] = c.x; v[1] = c.y; v[2] = c.z; v[3] = c.w;
        } else {
            for (int i = 0; i < 4; ++i)
                if (t0 + i < nT) v[i] = counts[t0 + i];
        }
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = (v[i] + (uint32_t)E - 1u) / (uint32_t)E * (uint32_t)E;
            mine += v[i];
        }
        uint32_t incl = mine;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            uint32_t s = wsum[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                uint32_t o = __shfl_up_sync(0xffffffffu, s, d);
                if (lane >= d) s += o;
            }
            wsum[lane] = s;   // inclusive over warps
        }
        __syncthreads();
        uint64_t prefix = carry_s + (warp > 0 ? wsum[warp - 1] : 0u) + incl - mine;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            prefix += v[i];
            if (t0 + i < nT) {
                if (prefix >= (1ull << 32)) us::set_status(status, US_ERR_TOO_LARGE);
                tile_off[t0 + i + 1] = (uint32_t)prefix;
            }
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry_s = prefix;
        __syncthreads();
    }
}

template <int ELEM>
__global__ void __launch_bounds__(kEncThreads)
enc_pack_kernel(const void* __restrict__ W, int64_t ldw, int TM, int TK, int nTK, int order,
                const uint64_t* __restrict__ bitmap, const uint32_t* __restrict__ tile_off,
                uint8_t* __restrict__ values, uint64_t values_cap, unsigned* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int t = blockIdx.x;
    const int tm = t / nTK, tk = t - tm * nTK;
    const int64_t corner = (int64_t)tm * TM * ldw + (int64_t)tk * TK;
    const int nw = TM * TK / 64;
    const int npos = TM * TK;
    constexpr int EB = (ELEM == US_F16) ? 2 : 1;       // bytes per compacted element in smem
    uint32_t* wpre = reinterpret_cast<uint32_t*>(smem);               // nw word prefixes
    uint8_t* cbuf = smem + ((nw * 4 + 15) & ~15);                     // compacted elements
    __shared__ uint32_t warp_tot[kEncThreads / 32];

    const uint64_t o0 = tile_off[t], o1 = tile_off[t + 1];
    const int bits = (ELEM == US_F16) ? 16 : (ELEM == US_I4 ? 4 : 2);
    if (o1 < o0 || o1 * bits > values_cap * 8) {
        if (threadIdx.x == 0) us::set_status(status, US_ERR_WORKSPACE);
        return;
    }
    const uint64_t* words = bitmap + (int64_t)t * nw;

    // exclusive prefix of the word popcounts (nw <= 512 = 2 per thread)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t c0 = 0, c1 = 0;
    const int w0 = 2 * threadIdx.x, w1 = w0 + 1;
    if (w0 < nw) c0 = __popcll(words[w0]);
    if (w1 < nw) c1 = __popcll(words[w1]);
    uint32_t incl = c0 + c1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
    for (int i = 0; i < warp; ++i) before += warp_tot[i];
    const uint32_t excl = before + incl - (c0 + c1);
    if (w0 < nw) wpre[w0] = excl;
    if (w1 < nw) wpre[w1] = excl + c0;
    uint32_t P = 0;
    for (int i = 0; i < kEncThreads / 32; ++i) P += warp_tot[i];
    __syncthreads();
    if (P > o1 - o0) {                       // cannot happen after enc_scan; guard anyway
        if (threadIdx.x == 0) us::set_status(status, US_ERR_CORRUPT);
        return;
    }

    // compact the set positions by rank
    for (int p = threadIdx.x; p < npos; p += kEncThreads) {
        const int w = p >> 6, b = p & 63;
        const uint64_t word = words[w];
        if ((word >> b) & 1ull) {
            const uint32_t rank = wpre[w] + __popcll(word & ((1ull << b) - 1ull));
            const int64_t idx = corner + pos_offset(order, TM, TK, p, ldw);
            if (ELEM == US_F16)
                reinterpret_cast<uint16_t*>(cbuf)[rank] = reinterpret_cast<const uint16_t*>(W)[idx];
            else
                cbuf[rank] = (uint8_t)reinterpret_cast<const int8_t*>(W)[idx] & (ELEM == US_I4 ? 0x0Fu : 0x03u);
        }
    }
    __syncthreads();

    // write the run [o0, o1) with zero padding, 16 bytes per thread-step
    const uint64_t run_bytes = (o1 - o0) * bits / 8;
    uint8_t* dst = values + o0 * bits / 8;
    for (uint64_t q = (uint64_t)threadIdx.x * 16; q < run_bytes; q += (uint64_t)kEncThreads * 16) {
        uint32_t v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            uint32_t word = 0;
#pragma unroll
            for (int bsub = 0; bsub < 4; ++bsub) {
                const uint64_t byte = q + r * 4 + bsub;
                uint32_t by = 0;
                if (ELEM == US_F16) {
                    const uint64_t e = byte >> 1;
                    if (e < P) {
                        const uint16_t h = reinterpret_cast<const uint16_t*>(cbuf)[e];
                        by = (byte & 1) ? (h >> 8) : (h & 0xFF);
                    }
                } else if (ELEM == US_I4) {
                    const uint64_t e0 = byte * 2, e1 = e0 + 1;
                    if (e0 < P) by |= cbuf[e0];
                    if (e1 < P) by |= (uint32_t)cbuf[e1] << 4;
                } else {                               // int2: four per byte, earlier lower
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (byte * 4 + u < P) by |= (uint32_t)cbuf[byte * 4 + u] << (2 * u);
                }
                word |= (by & 0xFFu) << (8 * bsub);
            }
            v[r] = word;
        }
        *reinterpret_cast<uint4*>(dst + q) = make_uint4(v[0], v[1], v[2], v[3]);
    }
    (void)EB;
}

// -------------------------------------- row-scan tiles 64 columns wide --
// Bit k of the result is set iff byte k of the 16 bytes is nonzero: for each
// word, (x & 0x7F..) + 0x7F.. carries into bit 7 of every byte whose low seven
// bits are not all zero; OR-ing x covers the top bit; the four byte flags
// (bits 0, 8, 16, 24 after the shift) are gathered into bits 24..27 by one
// multiplication by 2^24 + 2^17 + 2^10 + 2^3 (no two partial products share
// a bit below 28).
__device__ __forceinline__ uint32_t nz_bytes16(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t t = ((((w[r] & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w[r]) & 0x80808080u) >> 7;
        m |= ((t * 0x01020408u) >> 24) << (4 * r);
    }
    return m;
}
// Bit k set iff half k of the 8 halves is nonzero (+0 and -0 count as zero).
__device__ __forceinline__ uint32_t nz_halves8(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t t = (((w[r] & 0x7FFF7FFFu) + 0x7FFF7FFFu) & 0x80008000u) >> 15;   // bits 0 and 16
        m |= ((t | (t >> 15)) & 3u) << (2 * r);
    }
    return m;
}
// Nonzero if some byte of the 16 lies outside the code range [-lim, lim - 1]
// (lim = 8 for int4, 2 for int2): bytes + lim, added byte by byte, must stay
// below 2 lim.
__device__ __forceinline__ uint32_t out_of_range16(uint4 v, uint32_t lim) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t add = lim * 0x01010101u, bad = (~(2u * lim - 1u) & 0xFFu) * 0x01010101u;
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) r |= (((w[i] & 0x7F7F7F7Fu) + add) ^ (w[i] & 0x80808080u)) & bad;
    return r;
}

// ELEM's 16-byte loads: LPR lanes per tile row (64 elements), RPW rows per warp
template <int ELEM>
struct Row64 {
    static constexpr int kLPR = ELEM == US_F16 ? 8 : 4;
    static constexpr int kRPW = 32 / kLPR;
    static constexpr int kBPL = 64 / kLPR;          // mask bits per lane
    static constexpr int kEB = ELEM == US_F16 ? 2 : 1;
};

template <int ELEM>
__global__ void __launch_bounds__(kEncThreads)
enc_count_row64_kernel(const void* __restrict__ W, int64_t ldw, int TM, int nTK, uint64_t* __restrict__ bitmap,
                       uint32_t* __restrict__ counts, unsigned* status) {
    using R = Row64<ELEM>;
    const int t = blockIdx.x;
    const int tm = t / nTK, tk = t - tm * nTK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = lane % R::kLPR, rsub = lane / R::kLPR;
    const uint8_t* base = reinterpret_cast<const uint8_t*>(W) + ((int64_t)tm * TM * ldw + (int64_t)tk * 64) * R::kEB;
    __shared__ int warp_sum[kEncThreads / 32];
    int my = 0;
    for (int r0 = warp * R::kRPW; r0 < TM; r0 += (kEncThreads / 32) * R::kRPW) {
        const int row = r0 + rsub;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)row * ldw * R::kEB) + seg);
        const uint32_t m = ELEM == US_F16 ? nz_halves8(v) : nz_bytes16(v);
        if (ELEM != US_F16 && out_of_range16(v, ELEM == US_I4 ? 8u : 2u)) us::set_status(status, US_ERR_INVALID_ARG);
        uint64_t word = (uint64_t)m << (R::kBPL * seg);
#pragma unroll
        for (int d = 1; d < R::kLPR; d <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, d);
        if (seg == 0) bitmap[(int64_t)t * TM + row] = word;
        my += __popc(m);
    }
#pragma unroll
    for (int d = 16; d; d >>= 1) my += __shfl_xor_sync(0xffffffffu, my, d);
    if (lane == 0) warp_sum[warp] = my;
    __syncthreads();
    if (threadIdx.x == 0) {
        int sum = 0;
        for (int i = 0; i < kEncThreads / 32; ++i) sum += warp_sum[i];
        counts[t] = (uint32_t)sum;
    }
}

template <int ELEM>
__global__ void __launch_bounds__(kEncThreads)
enc_pack_row64_kernel(const void* __restrict__ W, int64_t ldw, int TM, int nTK, const uint64_t* __restrict__ bitmap,
                      const uint32_t* __restrict__ tile_off, uint8_t* __restrict__ values, uint64_t values_cap,
                      unsigned* status) {
    using R = Row64<ELEM>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int t = blockIdx.x;
    const int tm = t / nTK, tk = t - tm * nTK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = lane % R::kLPR, rsub = lane / R::kLPR;
    uint32_t* wpre = reinterpret_cast<uint32_t*>(smem);                // TM row prefixes
    uint8_t* cbuf = smem + TM * 4;                                     // compacted elements, 1 or 2 bytes each
    __shared__ uint32_t warp_tot[kEncThreads / 32];

    const uint64_t o0 = tile_off[t], o1 = tile_off[t + 1];
    const int bits = (ELEM == US_F16) ? 16 : (ELEM == US_I4 ? 4 : 2);
    if (o1 < o0 || o1 * bits > values_cap * 8 || o1 - o0 > (uint64_t)TM * 64) {
        if (threadIdx.x == 0) us::set_status(status, US_ERR_WORKSPACE);
        return;
    }
    const uint64_t* words = bitmap + (int64_t)t * TM;
    // exclusive prefix of the row popcounts (TM <= 256: one row a thread)
    const uint32_t c = threadIdx.x < TM ? (uint32_t)__popcll(words[threadIdx.x]) : 0u;
    uint32_t incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0, P = 0;
    for (int i = 0; i < kEncThreads / 32; ++i) {
        if (i < warp) before += warp_tot[i];
        P += warp_tot[i];
    }
    if (threadIdx.x < TM) wpre[threadIdx.x] = before + incl - c;
    const uint32_t run = (uint32_t)(o1 - o0);
    if (P > run) {                           // cannot happen after enc_scan; guard anyway
        if (threadIdx.x == 0) us::set_status(status, US_ERR_CORRUPT);
        return;
    }
    // the padding elements of the run are zero
    for (uint32_t e = P + threadIdx.x; e < run; e += kEncThreads) {
        if (ELEM == US_F16) reinterpret_cast<uint16_t*>(cbuf)[e] = 0;
        else cbuf[e] = 0;
    }
    __syncthreads();

    // each lane: its 16-byte piece of a row, its set elements to their ranks
    const uint8_t* base = reinterpret_cast<const uint8_t*>(W) + ((int64_t)tm * TM * ldw + (int64_t)tk * 64) * R::kEB;
    for (int r0 = warp * R::kRPW; r0 < TM; r0 += (kEncThreads / 32) * R::kRPW) {
        const int row = r0 + rsub;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)row * ldw * R::kEB) + seg);
        const uint64_t word = words[row];
        uint32_t m = (uint32_t)(word >> (R::kBPL * seg)) & ((1u << R::kBPL) - 1u);
        uint32_t rank = wpre[row] + (uint32_t)__popcll(word & ((1ull << (R::kBPL * seg)) - 1ull));
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
        while (m) {
            const int k = __ffs(m) - 1;
            m &= m - 1u;
            if (ELEM == US_F16) {
                reinterpret_cast<uint16_t*>(cbuf)[rank++] = (uint16_t)(vw[k >> 1] >> (16 * (k & 1)));
            } else {
                cbuf[rank++] = (uint8_t)((vw[k >> 2] >> (8 * (k & 3))) & (ELEM == US_I4 ? 0x0Fu : 0x03u));
            }
        }
    }
    __syncthreads();

    // write the run, 16 bytes per thread-step (the run is a whole number of 16 bytes)
    const uint32_t run_bytes = run * (uint32_t)bits / 8u;
    uint8_t* dst = values + o0 * bits / 8;
    for (uint32_t q = threadIdx.x * 16u; q < run_bytes; q += kEncThreads * 16u) {
        uint4 out;
        if (ELEM == US_F16) {
            out = *reinterpret_cast<const uint4*>(cbuf + q);
        } else if (ELEM == US_I4) {
            // 32 elements, one per byte -> 16 bytes of nibble pairs (earlier low)
            const uint4 a = *reinterpret_cast<const uint4*>(cbuf + 2 * q);
            const uint4 b = *reinterpret_cast<const uint4*>(cbuf + 2 * q + 16);
            auto pair2 = [](uint32_t x, uint32_t y) {
                return __byte_perm(x | (x >> 4), y | (y >> 4), 0x6420u);
            };
            out = make_uint4(pair2(a.x, a.y), pair2(a.z, a.w), pair2(b.x, b.y), pair2(b.z, b.w));
        } else {
            // 64 elements -> 16 bytes, four per byte (earlier lower)
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 a = *reinterpret_cast<const uint4*>(cbuf + 4 * q + 16 * i);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
                uint32_t word = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t x = aw[j];
                    word |= ((x | (x >> 6) | (x >> 12) | (x >> 18)) & 0xFFu) << (8 * j);
                }
                o[i] = word;
            }
            out = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(dst + q) = out;
    }
}

// ---------------------------------------------------- IE-BME with areas --
// UnionSparse section V-A with Q = RA*CA areas (Fig. 7): a TM x TK tile,
// after its optional row permutation, is cut into RA x CA areas of LM x LK;
// logical position (i, j) of the union mask is set iff some area holds a
// nonzero there; each set position emits one value per area, zeros included,
// at CV[o_t + q P_t + rho] with q = a*CA + c.
struct IeShape {
    int TM, TK, RA, CA, nTK;
};

// original row (within the tile) of row r of the reordered tile
__device__ __forceinline__ int ie_row(const uint8_t* perm, int64_t t, int TM, int r) {
    if (!perm) return r;
    const int v = perm[t * TM + r];
    return v < TM ? v : r;                  // out-of-range entries were reported by the count kernel
}

template <int ELEM>
__global__ void __launch_bounds__(kEncThreads)
enc_ie_count_kernel(const void* __restrict__ W, int64_t ldw, IeShape sh, const uint8_t* __restrict__ perm,
                    uint64_t* __restrict__ bitmap, uint32_t* __restrict__ counts, unsigned* status) {
    const int t = blockIdx.x;
    const int tm = t / sh.nTK, tk = t - tm * sh.nTK;
    const int LM = sh.TM / sh.RA, LK = sh.TK / sh.CA;
    const int nw = LM * LK / 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int warp_sum[kEncThreads / 32];
    __shared__ uint32_t seen[8];            // rows named by the permutation (TM <= 256)
    if (threadIdx.x < 8) seen[threadIdx.x] = 0;
    __syncthreads();
    if (perm && threadIdx.x < sh.TM) {
        const int v = perm[(int64_t)t * sh.TM + threadIdx.x];
        if (v >= sh.TM) us::set_status(status, US_ERR_INVALID_ARG);
        else atomicOr(&seen[v >> 5], 1u << (v & 31));
    }
    __syncthreads();
    if (perm && threadIdx.x == 0) {
        int n = 0;
        for (int i = 0; i < 8; ++i) n += __popc(seen[i]);
        if (n != sh.TM) us::set_status(status, US_ERR_INVALID_ARG);   // a row named twice
    }
    const int64_t row0 = (int64_t)tm * sh.TM;
    const int64_t col0 = (int64_t)tk * sh.TK;
    int my = 0;
    for (int w = warp; w < nw; w += kEncThreads / 32) {
        uint32_t half[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int lp = w * 64 + h * 32 + lane;
            const int i = lp / LK, j = lp - i * LK;
            bool any = false;
            for (int a = 0; a < sh.RA; ++a) {
                const int64_t r = row0 + ie_row(perm, t, sh.TM, a * LM + i);
                for (int c = 0; c < sh.CA; ++c) {
                    const int64_t idx = r * ldw + col0 + c * LK + j;
                    any |= is_nonzero<ELEM>(W, idx);
                    if (ELEM == US_I4) {
                        const int8_t v = reinterpret_cast<const int8_t*>(W)[idx];
                        if (v < -8 || v > 7) us::set_status(status, US_ERR_INVALID_ARG);
                    }
                }
            }
            half[h] = __ballot_sync(0xffffffffu, any);
        }
        if (lane == 0) {
            bitmap[(int64_t)t * nw + w] = (uint64_t)half[0] | ((uint64_t)half[1] << 32);
            my += __popc(half[0]) + __popc(half[1]);
        }
    }
    if (lane == 0) warp_sum[warp] = my;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int i = 0; i < kEncThreads / 32; ++i) s += warp_sum[i];
        counts[t] = (uint32_t)(s * sh.RA * sh.CA);              // the run holds Q * P_t values
    }
}

template <int ELEM>
__global__ void __launch_bounds__(kEncThreads)
enc_ie_pack_kernel(const void* __restrict__ W, int64_t ldw, IeShape sh, const uint8_t* __restrict__ perm,
                   const uint64_t* __restrict__ bitmap, const uint32_t* __restrict__ tile_off,
                   uint8_t* __restrict__ values, uint64_t values_cap, unsigned* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int t = blockIdx.x;
    const int tm = t / sh.nTK, tk = t - tm * sh.nTK;
    const int LM = sh.TM / sh.RA, LK = sh.TK / sh.CA, Q = sh.RA * sh.CA;
    const int lpos = LM * LK, nw = lpos / 64;
    uint32_t* wpre = reinterpret_cast<uint32_t*>(smem);
    uint8_t* cbuf = smem + ((nw * 4 + 15) & ~15);                     // Q * P compacted elements
    __shared__ uint32_t warp_tot[kEncThreads / 32];

    const uint64_t o0 = tile_off[t], o1 = tile_off[t + 1];
    const int bits = (ELEM == US_F16) ? 16 : 4;
    if (o1 < o0 || o1 * bits > values_cap * 8) {
        if (threadIdx.x == 0) us::set_status(status, US_ERR_WORKSPACE);
        return;
    }
    const uint64_t* words = bitmap + (int64_t)t * nw;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t c0 = 0, c1 = 0;
    const int w0 = 2 * threadIdx.x, w1 = w0 + 1;
    if (w0 < nw) c0 = __popcll(words[w0]);
    if (w1 < nw) c1 = __popcll(words[w1]);
    uint32_t incl = c0 + c1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
    for (int i = 0; i < warp; ++i) before += warp_tot[i];
    const uint32_t excl = before + incl - (c0 + c1);
    if (w0 < nw) wpre[w0] = excl;
    if (w1 < nw) wpre[w1] = excl + c0;
    uint32_t P = 0;
    for (int i = 0; i < kEncThreads / 32; ++i) P += warp_tot[i];
    __syncthreads();
    const uint32_t L = P * (uint32_t)Q;                              // values in the run
    if (L > o1 - o0) {
        if (threadIdx.x == 0) us::set_status(status, US_ERR_CORRUPT);
        return;
    }
    // each set logical position: one value per area, CV[o_t + q P + rho]
    const int64_t row0 = (int64_t)tm * sh.TM, col0 = (int64_t)tk * sh.TK;
    for (int lp = threadIdx.x; lp < lpos; lp += kEncThreads) {
        const int w = lp >> 6, b = lp & 63;
        const uint64_t word = words[w];
        if (!((word >> b) & 1ull)) continue;
        const uint32_t rank = wpre[w] + __popcll(word & ((1ull << b) - 1ull));
        const int i = lp / LK, j = lp - i * LK;
        for (int a = 0; a < sh.RA; ++a) {
            const int64_t r = row0 + ie_row(perm, t, sh.TM, a * LM + i);
            for (int c = 0; c < sh.CA; ++c) {
                const int64_t idx = r * ldw + col0 + c * LK + j;
                const uint32_t e = (uint32_t)(a * sh.CA + c) * P + rank;
                if (ELEM == US_F16)
                    reinterpret_cast<uint16_t*>(cbuf)[e] = reinterpret_cast<const uint16_t*>(W)[idx];
                else
                    cbuf[e] = (uint8_t)reinterpret_cast<const int8_t*>(W)[idx] & 0x0Fu;
            }
        }
    }
    __syncthreads();
    // the run [o0, o1) with zero padding, 16 bytes per thread-step
    const uint64_t run_bytes = (o1 - o0) * bits / 8;
    uint8_t* dst = values + o0 * bits / 8;
    for (uint64_t q = (uint64_t)threadIdx.x * 16; q < run_bytes; q += (uint64_t)kEncThreads * 16) {
        uint32_t v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            uint32_t word = 0;
#pragma unroll
            for (int bsub = 0; bsub < 4; ++bsub) {
                const uint64_t byte = q + r * 4 + bsub;
                uint32_t by = 0;
                if (ELEM == US_F16) {
                    const uint64_t e = byte >> 1;
                    if (e < L) {
                        const uint16_t h = reinterpret_cast<const uint16_t*>(cbuf)[e];
                        by = (byte & 1) ? (h >> 8) : (h & 0xFF);
                    }
                } else {
                    const uint64_t e0 = byte * 2, e1 = e0 + 1;
                    if (e0 < L) by |= cbuf[e0];
                    if (e1 < L) by |= (uint32_t)cbuf[e1] << 4;
                }
                word |= (by & 0xFFu) << (8 * bsub);
            }
            v[r] = word;
        }
        *reinterpret_cast<uint4*>(dst + q) = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

}  // namespace

namespace us {

size_t encode_pack_smem(int TM, int TK, int elem) {
    const int nw = TM * TK / 64;
    return (size_t)((nw * 4 + 15) & ~15) + (size_t)TM * TK * (elem == US_F16 ? 2 : 1);
}

// The 16-byte-load kernels: row scan, 64-column tiles, W and every row start
// 16-byte aligned.
template <int ELEM>
us_status launch_encode_row64(const void* W, int64_t ldw, int TM, int nTK, int64_t nT, uint64_t* bitmap,
                              uint32_t* tile_off, void* values, size_t values_cap, uint32_t* counts, unsigned* status,
                              cudaStream_t st) {
    enc_count_row64_kernel<ELEM><<<(unsigned)nT, kEncThreads, 0, st>>>(W, ldw, TM, nTK, bitmap, counts, status);
    if (cudaGetLastError() != cudaSuccess) return US_ERR_CUDA;
    enc_scan_kernel<<<1, 1024, 0, st>>>(counts, nT, ELEM == US_F16 ? 8 : (ELEM == US_I4 ? 32 : 64), tile_off, status);
    if (cudaGetLastError() != cudaSuccess) return US_ERR_CUDA;
    const size_t smem = (size_t)TM * 4 + (size_t)TM * 64 * (ELEM == US_F16 ? 2 : 1);
    if (cudaFuncSetAttribute(enc_pack_row64_kernel<ELEM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return US_ERR_CUDA;
    enc_pack_row64_kernel<ELEM><<<(unsigned)nT, kEncThreads, smem, st>>>(W, ldw, TM, nTK, bitmap, tile_off,
                                                                         (uint8_t*)values, values_cap, status);
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

us_status launch_encode(const void* W, int64_t ldw, int M, int K, int TM, int TK, int elem, int order,
                        uint64_t* bitmap, uint32_t* tile_off, void* values, size_t values_cap,
                        uint32_t* counts, unsigned* status, cudaStream_t st) {
    const int nTM = M / TM, nTK = K / TK;
    const int64_t nT = (int64_t)nTM * nTK;
    const int eb = elem == US_F16 ? 2 : 1;
    if (order == US_ORDER_ROW && TK == 64 && (reinterpret_cast<uintptr_t>(W) & 15u) == 0 && (ldw * eb) % 16 == 0) {
        if (elem == US_F16)
            return launch_encode_row64<US_F16>(W, ldw, TM, nTK, nT, bitmap, tile_off, values, values_cap, counts,
                                               status, st);
        if (elem == US_I4)
            return launch_encode_row64<US_I4>(W, ldw, TM, nTK, nT, bitmap, tile_off, values, values_cap, counts,
                                              status, st);
        return launch_encode_row64<US_I2>(W, ldw, TM, nTK, nT, bitmap, tile_off, values, values_cap, counts, status,
                                          st);
    }
    const size_t smem = encode_pack_smem(TM, TK, elem);
    if (elem == US_F16) {
        enc_count_kernel<US_F16><<<(unsigned)nT, kEncThreads, 0, st>>>(W, ldw, TM, TK, nTK, order, bitmap, counts,
                                                                      status);
    } else if (elem == US_I4) {
        enc_count_kernel<US_I4><<<(unsigned)nT, kEncThreads, 0, st>>>(W, ldw, TM, TK, nTK, order, bitmap, counts,
                                                                     status);
    } else {
        enc_count_kernel<US_I2><<<(unsigned)nT, kEncThreads, 0, st>>>(W, ldw, TM, TK, nTK, order, bitmap, counts,
                                                                     status);
    }
    if (cudaGetLastError() != cudaSuccess) return US_ERR_CUDA;
    enc_scan_kernel<<<1, 1024, 0, st>>>(counts, nT, elem == US_F16 ? 8 : (elem == US_I4 ? 32 : 64), tile_off, status);
    if (cudaGetLastError() != cudaSuccess) return US_ERR_CUDA;
    if (elem == US_F16) {
        if (cudaFuncSetAttribute(enc_pack_kernel<US_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return US_ERR_CUDA;
        enc_pack_kernel<US_F16><<<(unsigned)nT, kEncThreads, smem, st>>>(
            W, ldw, TM, TK, nTK, order, bitmap, tile_off, (uint8_t*)values, values_cap, status);
    } else if (elem == US_I4) {
        if (cudaFuncSetAttribute(enc_pack_kernel<US_I4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return US_ERR_CUDA;
        enc_pack_kernel<US_I4><<<(unsigned)nT, kEncThreads, smem, st>>>(
            W, ldw, TM, TK, nTK, order, bitmap, tile_off, (uint8_t*)values, values_cap, status);
    } else {
        if (cudaFuncSetAttribute(enc_pack_kernel<US_I2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return US_ERR_CUDA;
        enc_pack_kernel<US_I2><<<(unsigned)nT, kEncThreads, smem, st>>>(
            W, ldw, TM, TK, nTK, order, bitmap, tile_off, (uint8_t*)values, values_cap, status);
    }
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

us_status launch_encode_ie(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, int elem,
                           const uint8_t* perm, uint64_t* bitmap, uint32_t* tile_off, void* values,
                           size_t values_cap, uint32_t* counts, unsigned* status, cudaStream_t st) {
    IeShape sh{TM, TK, RA, CA, K / TK};
    const int64_t nT = (int64_t)(M / TM) * (K / TK);
    const size_t smem = encode_pack_smem(TM, TK, elem);             // Q * P <= TM * TK elements
    if (elem == US_F16)
        enc_ie_count_kernel<US_F16><<<(unsigned)nT, kEncThreads, 0, st>>>(W, ldw, sh, perm, bitmap, counts, status);
    else
        enc_ie_count_kernel<US_I4><<<(unsigned)nT, kEncThreads, 0, st>>>(W, ldw, sh, perm, bitmap, counts, status);
    if (cudaGetLastError() != cudaSuccess) return US_ERR_CUDA;
    enc_scan_kernel<<<1, 1024, 0, st>>>(counts, nT, elem == US_F16 ? 8 : 32, tile_off, status);
    if (cudaGetLastError() != cudaSuccess) return US_ERR_CUDA;
    if (elem == US_F16) {
        if (cudaFuncSetAttribute(enc_ie_pack_kernel<US_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return US_ERR_CUDA;
        enc_ie_pack_kernel<US_F16><<<(unsigned)nT, kEncThreads, smem, st>>>(W, ldw, sh, perm, bitmap, tile_off,
                                                                            (uint8_t*)values, values_cap, status);
    } else {
        if (cudaFuncSetAttribute(enc_ie_pack_kernel<US_I4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return US_ERR_CUDA;
        enc_ie_pack_kernel<US_I4><<<(unsigned)nT, kEncThreads, smem, st>>>(W, ldw, sh, perm, bitmap, tile_off,
                                                                           (uint8_t*)values, values_cap, status);
    }
    return cudaGetLastError() == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace us
