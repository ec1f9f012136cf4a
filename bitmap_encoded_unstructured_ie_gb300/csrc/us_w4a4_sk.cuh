// us_w4a4_sk.cuh -- W4A4 bitmap SpMM for 1..32 tokens, the tile sequence spread
// evenly over the SMs: the kernel template and its shared-memory plan, for
// the translation units that instantiate it (us_w4a4_sk.cu: plain tiles).
//
// Y = W . X with W int4 in 64 x 64 bitmap tiles, row-major scan (IE-BME of
// "UnionSparse: An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM
// Inference on Edge", section V-A, one area), X int4 per token, int32
// accumulation and the dequantised fp16 epilogue of the same page's Fig. 2.
//
// Decode-sized products move a few MB per call, so the kernel is built around
// latency, not around a steady stream:
//  * balanced partition: CTA c of G owns the tiles [c*nT/G, (c+1)*nT/G) of the
//    tile sequence t = tm*nTK + tk (one CTA per SM, a second one of the next
//    launch fits beside it).  A contiguous run of tiles is contiguous in the
//    bitmap and in the value array, so one chunk of four tiles arrives with two
//    1-D bulk copies (TMA), packed into a byte ring by their real length;
//  * decode once into dense tiles: a warp turns a tile into 64 x 64 packed int4
//    in shared memory (lane l: rows l and l + 32; row bases from one warp scan
//    of packed popcounts, the word-level part of UnionSparse's idx_base,
//    section VI-B; a byte-step per eight positions: selector table + PRMT).
//    Weights flagged static are decoded this way BEFORE the dependency wait,
//    while the previous launch still runs; after it only the multiply is left
//    (dp4a for up to 7 tokens, mma.sync in 8-token blocks above that).  Tiles
//    beyond the dense slots, and all tiles of non-static weights, are decoded
//    after the wait into the warp's own slot;
//  * after the wait each warp fetches the activation slices of its own tiles
//    and goes on by itself;
//  * a band split between CTAs is finished by the CTA holding its first tile:
//    the others post their partial sums as 64-bit {value, tag} words (one
//    relaxed store each, no fence, no counter: the tag arrives with its value)
//    and the owner waits for the tags (bounded), adds, and clears them for the
//    next call.  Partials are integers, so the sum is exact in any order.
#pragma once
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kTM = 64, kTK = 64;
constexpr int kBm = kTM * kTK / 8;          // bitmap bytes per tile
constexpr int kValCap = kTM * kTK / 2;      // value bytes per tile, worst case
constexpr int kC = 4;                       // tiles per chunk
constexpr int kR = 16;                      // chunks in flight at most (mbarrier pairs)
// Two consumers share the kernel: NT == 0 multiplies N tokens with dp4a; NT > 0
// feeds mma.sync (fp16, fp32 accumulation) with NT blocks of eight tokens.
// Consumer warps: as many as two CTAs per SM can hold with every accumulator
// in registers.
__host__ __device__ constexpr int nw_for(int N, int NT) {
    return NT ? (NT == 1 ? 14 : (NT == 2 ? 10 : 6)) : (N == 1 ? 16 : (N <= 3 ? 14 : 12));
}
// consumer warps, then the weight producer warp, then the activation warp
__host__ __device__ constexpr int threads_for(int N, int NT) { return (nw_for(N, NT) + 2) * 32; }
__host__ __device__ constexpr int ntok_for(int N, int NT) { return NT ? 8 * NT : N; }   // token slots
constexpr int kLutRep = 4;                  // selector table replicas (bank spreading)
constexpr int kHeader = 512;
constexpr int kLutBytes = 256 * kLutRep * 8;   // {selector pair, odd-rank mask} per entry
constexpr int kSlot = kTM * kTK / 2;        // one decoded tile: 64 x 64 packed int4
constexpr int kMinRing = 2 * kC * (kBm + kValCap);   // at least two worst-case chunks
// IE-BME areas: a 64 x 64 super-tile is four 16 x 64 local tiles (sub-bands
// i = 0..3 of the 64-row band), each with a union mask of 128 / Q bytes, a
// 16-byte row permutation and a run of Q * P_t values (at most 1024 nibbles)
constexpr int kIeLocalRows = 16;
constexpr int kIeChunkCap = kC * 4 * (128 + 16 + 512);
constexpr int kMinRingIe = 2 * kIeChunkCap;

struct SkSmem {
    uint64_t full[kR], empty[kR];
    uint64_t xfull;                         // the activation copies have landed
    uint64_t xfull2;                        // those of a K range's wrapped part have landed
    uint32_t pos[kR];                       // ring offset of the chunk in slot s
    uint32_t bad[kR];                       // its offsets failed the checks
    uint32_t abort;
    uint32_t x2;                            // copies of a wrapped part were issued
    // this CTA's tile range [t0, t1), its first band, its band count, the
    // highest CTA sharing its last band, and t0's K tile: worked out once by
    // thread 0 (divisions by launch values), read by all after the barrier
    int t0, t1, band0, nb, c_hi, tk0;
};
static_assert(sizeof(SkSmem) <= kHeader, "header");

__host__ __device__ inline int sk_cta_of(int64_t t, int G, int nT) { return (int)(((t + 1) * G - 1) / nT); }
__host__ __device__ inline int sk_start(int c, int G, int nT) { return (int)((int64_t)c * nT / G); }

// Selector table entries {selector pair, odd-rank mask | popcount} for both
// consumers, generated at compile time (mma: 1).  The selectors move rank r
// to position p (make_sel); the consumer asks for a position order.  The dp4a
// consumer takes (p0 p2 p4 p6 | p1 p3 p5 p7), which packs the positions in the
// order of the packed activations (position 2i low, 2i + 1 high in byte i);
// the mma one (p0 p4 p1 p5 | p2 p6 p3 p7), the nibble order that its fp16
// conversion pairs up.  Clear positions take rank 7's byte, which the
// odd-rank mask empties unless all eight positions are set.  Only high
// nibbles of the odd/even bytes reach the dense word, so the mask's lowest
// nibble carries the byte's popcount (POPC issues at a quarter of the
// logic-op rate on this GPU; this costs one AND).
struct SelEntry { uint32_t sel, mask; };
struct SelTable { SelEntry e[2][256]; };
constexpr SelTable build_sel_table() {
    SelTable t{};
    for (int mma = 0; mma < 2; ++mma)
        for (uint32_t e = 0; e < 256; ++e) {
            const uint32_t sel = us::make_sel(e);
            uint32_t ps = 0, pop = 0;
            for (int i = 0; i < 8; ++i) {
                const int to = mma ? ((i & 3) * 2 + (i >> 2)) : ((i & 1) * 4 + (i >> 1));
                ps |= ((sel >> (4 * i)) & 0xFu) << (4 * to);
                pop += (e >> i) & 1u;
            }
            t.e[mma][e].sel = ps;
            t.e[mma][e].mask = (e == 255 ? 0xF0F0F0F0u : 0x00F0F0F0u) | pop;
        }
    return t;
}
__device__ const SelTable kSelTable = build_sel_table();


// Eight int2 values (low 16 bits, the earlier value in the lower bits) as
// eight sign-extended int4 nibbles: spread the 2-bit fields 8, 4 and 2 bits
// apart, then copy each sign bit into the two bits above it.
__device__ __forceinline__ uint32_t int2x8_to_int4x8(uint32_t x) {
    x &= 0xFFFFu;
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    x = (x | (x << 2)) & 0x33333333u;
    const uint32_t sgn = x & 0x22222222u;
    return x | (sgn << 1) | (sgn << 2);
}

// WB: weight bits (4: W4A4, 2: W2A4; the dense tiles hold int4 either way).
// IE: the tiles are 64 x 64 super-tiles of IE-BME 16 x 64 local tiles with
// p.ie_ra x p.ie_ca areas (p.ie_ca <= 2) and optional row permutations;
// p.nTM counts 64-row bands.
template <int N, int NT, int WB, bool IE = false>
__global__ void __launch_bounds__(threads_for(N, NT), 2)   // two per SM: this launch and the next
w4a4_sk_kernel(const UsKParams p) {
    constexpr int kNW = nw_for(N, NT);
    constexpr int kThreads = threads_for(N, NT);
    constexpr int NTOK = ntok_for(N, NT);
    constexpr int XROW = kTK / 2;               // staged activation bytes per K tile (packed int4)
    // 16 or more tokens: a wrapped K range's copies land on a barrier of their
    // own (measured: 4096 x 4096, N = 16: 7.68 -> 7.49 us; N = 8: 6.11 -> 6.15)
    constexpr bool kSplitX = NT >= 2;
    extern __shared__ __align__(128) uint8_t smem[];
    SkSmem& S = *reinterpret_cast<SkSmem*>(smem);
    uint2* lut = reinterpret_cast<uint2*>(smem + kHeader);
    // dense tiles (sk_slots x kSlot) follow the table, then the byte ring
    uint8_t* ring = smem + kHeader + kLutBytes + (size_t)p.sk_slots * kSlot;
    const uint32_t D = (uint32_t)p.sk_ring;
    const int nT = p.nTM * p.nTK, G = p.sk_grid;
    const int cta = blockIdx.x;
    // tile offsets: per + 1 of them; IE: per super-tile and sub-band the start
    // and end of the local tile's run, offs[8 q + 2 i + e]
    uint32_t* offs = reinterpret_cast<uint32_t*>(ring + D);
    // activations as given (packed int4): NTOK x xcols x XROW bytes; column xq of
    // token n holds K tile tk, where xq = tk when the CTAs span whole band
    // widths (xcols == nTK), else xq = the tile's place in the CTA's range
    int8_t* xs = reinterpret_cast<int8_t*>(offs + (IE ? p.sk_per * 8 : ((p.sk_per + 1 + 3) & ~3)));
    int* accs = reinterpret_cast<int*>(xs + NTOK * p.sk_xcols * XROW);          // bands x NTOK x 64
    uint16_t* sws = reinterpret_cast<uint16_t*>(accs + p.sk_nb * NTOK * kTM);     // bands x 64 row scales
    uint16_t* sxs = sws + p.sk_nb * kTM;                                          // NTOK token scales
    // per tile of the range: its band (relative to band0) << 16 | its K tile,
    // bit 15 set on a warp's first tile that waits for a wrapped K range
    uint32_t* tinfo = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(sws) +
                                                  (((size_t)p.sk_nb * kTM + NTOK) * 2 + 15) / 16 * 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool early = (p.flags & US_BITMAP_STATIC) != 0;   // weights may be fetched before the wait
    constexpr uint32_t kQ = 128u / WB;                      // elements per 16 bytes (run padding)
    constexpr int kLogEPW = WB == 4 ? 3 : 4;                // elements per 32-bit word: 8 or 16

    if (threadIdx.x == 0) {
        for (int i = 0; i < kR; ++i) {
            us::mbar_init(&S.full[i], 1);
            us::mbar_init(&S.empty[i], kC);                  // one arrival per tile
        }
        us::mbar_init(&S.xfull, 1);
        us::mbar_init(&S.xfull2, 1);
        S.abort = 0;
        S.x2 = 0;
        // 32-bit divisions while G x nT fits (below 28 M tiles), else 64-bit
        const bool n32 = (uint64_t)nT * (uint64_t)(G + 1) < (1ull << 32);
        const int a = n32 ? (int)((uint32_t)cta * (uint32_t)nT / (uint32_t)G) : sk_start(cta, G, nT);
        const int b = n32 ? (int)((uint32_t)(cta + 1) * (uint32_t)nT / (uint32_t)G) : sk_start(cta + 1, G, nT);
        const int ba = (int)((uint32_t)a / (uint32_t)p.nTK), bz = (int)((uint32_t)(b - 1) / (uint32_t)p.nTK);
        const int tl = (bz + 1) * p.nTK - 1;                  // last tile of the last band
        S.t0 = a;
        S.t1 = b;
        S.band0 = ba;
        S.nb = bz - ba + 1;
        S.c_hi = n32 ? (int)((((uint32_t)tl + 1u) * (uint32_t)G - 1u) / (uint32_t)nT) : sk_cta_of(tl, G, nT);
        S.tk0 = a - ba * p.nTK;
        us::fence_mbar_init();
    }
    for (int i = threadIdx.x; i < p.sk_nb * NTOK * kTM; i += kThreads) accs[i] = 0;
    __syncthreads();
    const int t0 = S.t0, t1 = S.t1, per = t1 - t0, band0 = S.band0, nb = S.nb;
    us::pdl_launch_dependents();

    int issued = 0, tail = 0;                                 // producer bookkeeping (lane 0)
    if (warp == kNW) {
        // ------------------------------------------------------------ producer
        if (!early) us::pdl_wait();
        if constexpr (IE) {
            // start and end of every local tile's run: four sub-bands per super-tile
            for (int idx = lane; idx < per * 8; idx += 32) {
                const uint32_t t = (uint32_t)(t0 + (idx >> 3)), b = t / (uint32_t)p.nTK;
                const uint64_t lt = (uint64_t)(4u * b + ((idx >> 1) & 3)) * p.nTK + (t - b * (uint32_t)p.nTK);
                offs[idx] = p.tile_off[lt + (idx & 1)];
            }
        } else {
            // the whole range heads for L2 at once; the ring then refills from there
            if (early && lane == 0) us::bulk_prefetch_l2(p.bitmap + (int64_t)t0 * (kBm / 8), (uint32_t)per * kBm);
            for (int i = lane; i <= per; i += 32) offs[i] = p.tile_off[t0 + i];
        }
        __syncwarp();
        if (!IE && early && lane == 0 && offs[per] > offs[0] && (offs[0] & (kQ - 1u)) == 0 &&
            (offs[per] & (kQ - 1u)) == 0 && (uint64_t)offs[per] * WB <= p.values_bytes * 8ull)
            us::bulk_prefetch_l2(p.values + offs[0] * WB / 8u, (offs[per] - offs[0]) * WB / 8u);
        const int nch = (per + kC - 1) / kC;
        uint32_t pos = 0;                                     // end of the newest chunk in the ring
        bool waited = !early;
        // lane 0: room for sz bytes of chunk ch.  The ring holds the chunks
        // [tail, ch) in order, from the start of chunk `tail` to `pos`, wrapping
        // at D.  False when a wait for the consumers gave up.
        auto place_chunk = [&](int ch, uint32_t sz, uint32_t& place) -> bool {
            for (;;) {
                const int inflight = ch - tail;
                if (inflight == 0) { place = 0; return true; }
                if (inflight < kR) {
                    const uint32_t s0 = S.pos[tail % kR];
                    if (pos > s0) {
                        if (pos + sz <= D) { place = pos; return true; }
                        if (sz <= s0) { place = 0; return true; }
                    } else if (pos + sz <= s0) {
                        place = pos;
                        return true;
                    }
                }
                // the consumers release a chunk before the previous launch has
                // finished only if all its tiles are decoded early: else wait
                // for that launch too before a bounded wait on them
                if (!waited && min((tail + 1) * kC, per) > p.sk_pre) {
                    us::pdl_wait();
                    waited = true;
                }
                if (!us::mbar_wait(&S.empty[tail % kR], (uint32_t)(tail / kR) & 1u, p.status)) return false;
                ++tail;
            }
        };
        for (int ch = 0; ch < nch; ++ch) {
            const int q0 = ch * kC, ct = min(kC, per - q0), slot = ch % kR;
            int fail = 0;
            if constexpr (IE) {
                // up to two parts (the chunk may cross into the next band) x four
                // sub-bands x {union masks, permutations, value runs}: lane
                // L = 8 kind + 4 part + sub-band issues one copy; the copies sit in
                // the ring in lane order
                const int Q = p.ie_ra * p.ie_ca;
                const uint32_t ub = 128u / (uint32_t)Q;       // union-mask bytes per local tile
                const uint32_t tq = (uint32_t)(t0 + q0), b0 = tq / (uint32_t)p.nTK;
                const int c0 = (int)(tq - b0 * (uint32_t)p.nTK);
                const int n0 = min(ct, p.nTK - c0);           // super-tiles in the first band
                const int kind = lane >> 3, pp = (lane >> 2) & 1, i = lane & 3;
                const int cnt = pp ? ct - n0 : n0, qf = q0 + (pp ? n0 : 0);
                const uint64_t lt = (uint64_t)(4u * (b0 + (uint32_t)pp) + (uint32_t)i) * p.nTK + (pp ? 0 : c0);
                bool ok = true;
                uint32_t a = 0, e = 0;
                if (kind == 2 && cnt > 0) {
                    a = offs[8 * qf + 2 * i];
                    e = offs[8 * (qf + cnt - 1) + 2 * i + 1];
                    for (int k = 0; k < cnt; ++k) {
                        const uint32_t s0 = offs[8 * (qf + k) + 2 * i], s1 = offs[8 * (qf + k) + 2 * i + 1];
                        ok = ok && s1 >= s0 && s1 - s0 <= 1024u && (s0 & 31u) == 0 && (s1 & 31u) == 0 && s0 >= a &&
                             s1 <= e && (uint64_t)s1 * 4u <= p.values_bytes * 8ull;
                    }
                }
                const bool all_ok = __all_sync(0xffffffffu, ok);
                uint32_t bytes = 0;
                const uint8_t* src = nullptr;
                if (lane < 24 && cnt > 0) {
                    if (kind == 0) {
                        bytes = (uint32_t)cnt * ub;
                        src = reinterpret_cast<const uint8_t*>(p.bitmap) + lt * ub;
                    } else if (kind == 1) {
                        bytes = p.perm ? (uint32_t)cnt * 16u : 0u;
                        src = p.perm ? p.perm + lt * 16u : nullptr;
                    } else {
                        bytes = all_ok ? (e - a) / 2u : 0u;
                        src = p.values + a / 2u;
                    }
                }
                uint32_t incl = bytes;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += o;
                }
                const uint32_t sz = __shfl_sync(0xffffffffu, incl, 31);
                uint32_t place = 0;
                if (lane == 0) {
                    if (!place_chunk(ch, sz, place)) {
                        fail = 1;
                    } else {
                        if (!all_ok) us::set_status(p.status, US_ERR_CORRUPT);
                        S.pos[slot] = place;
                        S.bad[slot] = all_ok ? 0u : 1u;
                        us::mbar_arrive_expect_tx(&S.full[slot], sz);
                    }
                }
                fail = __shfl_sync(0xffffffffu, fail, 0);
                place = __shfl_sync(0xffffffffu, place, 0);
                if (!fail) {
                    __syncwarp();
                    if (bytes) us::bulk_g2s(ring + place + (incl - bytes), src, bytes, &S.full[slot]);
                    if (lane == 0) {
                        for (int k = ct; k < kC; ++k) us::mbar_arrive(&S.empty[slot]);
                        pos = place + sz;
                        issued = ch + 1;
                    }
                    pos = __shfl_sync(0xffffffffu, pos, 0);
                }
            } else {
            bool ok = true;
            if (lane < ct) {
                const uint32_t a = offs[q0 + lane], e = offs[q0 + lane + 1];
                ok = e >= a && (e - a) <= (uint32_t)(kTM * kTK) && (a & (kQ - 1u)) == 0 && (e & (kQ - 1u)) == 0 &&
                     (uint64_t)e * WB <= p.values_bytes * 8ull;
            }
            const bool all_ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) {
                const uint32_t vb = all_ok ? (offs[q0 + ct] - offs[q0]) * WB / 8u : 0u;
                const uint32_t sz = (uint32_t)ct * kBm + vb;
                uint32_t place = 0;
                if (!place_chunk(ch, sz, place)) {
                    fail = 1;
                } else {
                    if (!all_ok) us::set_status(p.status, US_ERR_CORRUPT);
                    S.pos[slot] = place;
                    S.bad[slot] = all_ok ? 0u : 1u;
                    us::mbar_arrive_expect_tx(&S.full[slot], sz);
                    us::bulk_g2s(ring + place, p.bitmap + (int64_t)(t0 + q0) * (kBm / 8), (uint32_t)ct * kBm,
                                 &S.full[slot]);
                    if (vb) us::bulk_g2s(ring + place + ct * kBm, p.values + offs[q0] * WB / 8u, vb, &S.full[slot]);
                    // a short last chunk has fewer tiles: arrive for the missing ones
                    for (int i = ct; i < kC; ++i) us::mbar_arrive(&S.empty[slot]);
                    pos = place + sz;
                    issued = ch + 1;
                }
            }
            }
            if (__shfl_sync(0xffffffffu, fail, 0)) {
                S.abort = 1;
                break;
            }
        }
        if (!waited) us::pdl_wait();                          // idle now: take it off the epilogue's path
    } else if (warp == kNW + 1) {
        // ---------------------------------------------------------- activations
        // copied in as soon as the previous launch has finished, whatever the
        // weight producer and the consumers are still busy with
        us::pdl_wait();
        const bool all_k = p.sk_xcols == p.nTK;
        const int ncols = all_k ? p.nTK : per;
        const uint8_t* xg = reinterpret_cast<const uint8_t*>(p.X);
        const int tk0 = all_k ? 0 : S.tk0;
        const int len1 = min(ncols, p.nTK - tk0);            // the range may wrap past the band's end
        // with kSplitX a wrapped part (the next band's first K tiles) lands on a
        // barrier of its own: the copy engine takes the copies one after
        // another, the first part's go first, and the consumers reach the
        // wrapped part's tiles last
        uint64_t* bar2 = kSplitX ? &S.xfull2 : &S.xfull;
        if (lane == 0) {
            us::mbar_arrive_expect_tx(&S.xfull, (uint32_t)(p.N * (kSplitX ? len1 : ncols) * XROW));
            if (kSplitX && len1 < ncols) {
                S.x2 = 1;
                us::mbar_arrive_expect_tx(&S.xfull2, (uint32_t)(p.N * (ncols - len1) * XROW));
            }
        }
        __syncwarp();
        for (int n = lane; n < p.N; n += 32)
            us::bulk_g2s(xs + (int64_t)n * p.sk_xcols * XROW, xg + (int64_t)n * (p.K / 2) + (int64_t)tk0 * XROW,
                         (uint32_t)len1 * XROW, &S.xfull);
        if (len1 < ncols)
            for (int n = lane; n < p.N; n += 32)
                us::bulk_g2s(xs + ((int64_t)n * p.sk_xcols + len1) * XROW, xg + (int64_t)n * (p.K / 2),
                             (uint32_t)(ncols - len1) * XROW, bar2);
        if (p.Y)
            for (int n = lane; n < p.N; n += 32) sxs[n] = p.s_x[n];
    }
    else {
        // ----------------------------------------------------------- consumers
        // selector table (16 w form: d0's bytes become the low nibbles of a
        // packed word, d1's the high ones), kLutRep copies for bank spreading
        for (int e = threadIdx.x; e < 256; e += kNW * 32) {
            const SelEntry v = kSelTable.e[NT ? 1 : 0][e];
            const uint2 ent = make_uint2(v.sel, v.mask);
#pragma unroll
            for (int r = 0; r < kLutRep; ++r) lut[e * kLutRep + r] = ent;
        }
        // the padding tokens of the mma consumer multiply as zeros
        if (NTOK > p.N) {
            uint4* z = reinterpret_cast<uint4*>(xs + (int64_t)p.N * p.sk_xcols * XROW);
            const int nz = (NTOK - p.N) * p.sk_xcols * XROW / 16;
            for (int i = threadIdx.x; i < nz; i += kNW * 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        // static weights: their row scales are fixed too
        if (p.Y && early)
            for (int i = threadIdx.x; i < nb * kTM; i += kNW * 32) sws[i] = p.s_w[band0 * kTM + i];
        {
            // tiles from xsplit on read the wrapped part of the K range; bit 15
            // marks each warp's first such tile, where it waits for that part
            const int xsplit = kSplitX && p.sk_xcols != p.nTK ? min(per, p.nTK - S.tk0) : per;
            for (int i = threadIdx.x; i < per; i += kNW * 32) {
                const uint32_t t = (uint32_t)(t0 + i), b = t / (uint32_t)p.nTK;
                const bool first2 = i >= xsplit && i - kNW < xsplit;
                tinfo[i] = ((b - (uint32_t)band0) << 16) | (first2 ? 0x8000u : 0u) | (t - b * (uint32_t)p.nTK);
            }
        }
        us::named_bar_sync(1, kNW * 32);

        const uint32_t lut_lane = (uint32_t)(lane % kLutRep);
        // tiles decoded before the wait: the plan's count, capped at this CTA's
        // own range (ranges differ by one tile where G does not divide nT)
        const int P = early ? min(p.sk_pre, per) : 0;
        // Decode tile q of the range into the dense packed-int4 tile dst: lane l
        // takes rows l and l + 32; row bases come from one warp scan of packed
        // popcounts (the word-level part of UnionSparse's idx_base, section
        // VI-B); a byte-step turns eight positions into one word of eight
        // nibbles.  False when the wait for the tile's chunk gave up.
        auto decode_tile = [&](int q, uint8_t* dst) -> bool {
            const int ch = q / kC, slot = ch % kR;
            if (!us::mbar_wait(&S.full[slot], (uint32_t)(ch / kR) & 1u, p.status)) {
                S.abort = 1;
                return false;
            }
            const int ct = min(kC, per - ch * kC);
            const uint8_t* base = ring + S.pos[slot];
            if constexpr (IE) {
                // four 16 x 64 local tiles (sub-bands i), each with Q areas.  Lane
                // work item: 32-bit union-mask word w32 = lane / Q (union row u,
                // segment sg of it) of area qa = lane % Q, i.e. 32 positions of
                // reordered row r = (qa / CA) LM + u, columns 32 (half) ..; the
                // value of the position of union rank rho in area qa is element
                // qa P_t + rho of the local tile's run (UnionSparse, section V-A)
                const int Q = p.ie_ra * p.ie_ca, CA = p.ie_ca;
                const int LM = kIeLocalRows / p.ie_ra, spr = 2 / CA;   // union rows, words per row
                const int nwq = 32 / Q;                                  // union words per local tile
                const uint32_t ub = 128u / (uint32_t)Q;
                const bool hasperm = p.perm != nullptr, bad = S.bad[slot] != 0;
                const int q0 = ch * kC;
                const int n0 = min(ct, p.nTK - (int)(tinfo[q0] & 0x7FFFu));   // super-tiles in the first band
                const int pp = (q - q0) < n0 ? 0 : 1;
                const int qf = q0 + (pp ? n0 : 0), cnt = pp ? ct - n0 : n0, kq = q - qf;
                // the chunk's value runs, lane j < 8 = (part j / 4, sub-band j % 4),
                // follow its union masks and permutations in that order
                uint32_t vbj = 0;
                if (lane < 8 && !bad) {
                    const int jp = lane >> 2, ji = lane & 3;
                    const int jc = jp ? ct - n0 : n0, jf = q0 + (jp ? n0 : 0);
                    if (jc > 0) vbj = (offs[8 * (jf + jc - 1) + 2 * ji + 1] - offs[8 * jf + 2 * ji]) / 2u;
                }
                uint32_t vinc = vbj;
#pragma unroll
                for (int d = 1; d < 8; d <<= 1) {
                    const uint32_t o = __shfl_up_sync(0xffffffffu, vinc, d);
                    if (lane >= d) vinc += o;
                }
                const uint32_t vexcl = vinc - vbj;
                const uint32_t vhead = (uint32_t)(4 * ct) * (ub + (hasperm ? 16u : 0u));
                const int qa = lane % Q, w32 = lane / Q;
                const int u = w32 / spr, sgm = w32 - u * spr;
                const int ra = qa / CA, ca = qa - ra * CA;
                const int r = ra * LM + u, half = ca * spr + sgm;
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    const uint32_t li = (uint32_t)((pp ? 4 * n0 : 0) + i * cnt + kq);   // place among the chunk's local tiles
                    const uint32_t* bm32 = reinterpret_cast<const uint32_t*>(base + li * ub);
                    const uint32_t s_q = offs[8 * q + 2 * i], e_q = offs[8 * q + 2 * i + 1];
                    const uint32_t vrun = __shfl_sync(0xffffffffu, vexcl, pp * 4 + i);
                    const uint32_t voff = vhead + vrun + (bad ? 0u : (s_q - offs[8 * qf + 2 * i]) / 2u);
                    const uint32_t* vw = reinterpret_cast<const uint32_t*>(base + voff);
                    const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(vw);
                    // union ranks: exclusive prefix of the words' popcounts
                    const uint32_t pc = lane < nwq ? (uint32_t)__popc(bm32[lane]) : 0u;
                    uint32_t inc = pc;
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const uint32_t o = __shfl_up_sync(0xffffffffu, inc, d);
                        if (lane >= d) inc += o;
                    }
                    const uint32_t Pt = __shfl_sync(0xffffffffu, inc, nwq - 1);
                    const uint32_t rho = __shfl_sync(0xffffffffu, inc - pc, w32);
                    const bool good = !bad && (uint32_t)Q * Pt <= e_q - s_q;
                    if (!good && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
                    const uint32_t word = good ? bm32[w32] : 0u;      // a bad tile decodes as zeros
                    uint32_t ob = (uint32_t)qa * Pt + rho, wi = ob >> 3;
                    uint32_t cur = vw[wi], nxt = vw[wi + 1], nn = vw[wi + 2];
                    uint32_t pw[4];
#pragma unroll
                    for (int bt = 0; bt < 4; ++bt) {
                        const uint32_t bb = __byte_perm(word, 0u, 0x4440u | (uint32_t)bt);
                        if (bt > 0) {
                            const uint32_t nwi = ob >> 3;
                            const uint32_t adv = nwi != wi;
                            cur = adv ? nxt : cur;
                            nxt = adv ? nn : nxt;
                            us::lds_u32_if(nn, adv, vbase + 4u * (nwi + 2u));
                            wi = nwi;
                        }
                        const uint32_t win = __funnelshift_r(cur, nxt, ob << 2);
                        const uint2 ent = lut[bb * kLutRep + lut_lane];
                        const uint32_t odd = win & ent.y, even = win << 4;
                        const uint32_t d0 = __byte_perm(even, odd, ent.x);
                        const uint32_t d1 = __byte_perm(even, odd, ent.x >> 16);
                        pw[bt] = us::lop3<us::kLopMux>(d0 >> 4, 0x0F0F0F0Fu, d1);
                        ob += ent.y & 0xFu;
                    }
                    // the reordered row's place in the original local tile
                    uint32_t orow = (uint32_t)r;
                    if (hasperm) {
                        const uint32_t v = base[4u * ct * ub + li * 16u + (uint32_t)r];
                        if (v < 16u) orow = v;
                        else us::set_status(p.status, US_ERR_CORRUPT);   // not a row of the tile
                    }
                    const int R = kIeLocalRows * i + (int)orow;
                    if constexpr (NT == 0) {
                        const int sw = (R >> 2) & 1;
                        *reinterpret_cast<uint4*>(dst + R * 32 + 16 * (half ^ sw)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    } else {
                        const int mb = R >> 4, g = R & 7, hr = (R >> 3) & 1;
#pragma unroll
                        for (int tt = 0; tt < 2; ++tt) {
                            const int sg = mb * 32 + g * 4 + 2 * half + tt;
                            const int ph = sg ^ ((sg >> 3) & 3);
                            *reinterpret_cast<uint2*>(dst + ph * 16 + hr * 8) = make_uint2(pw[2 * tt], pw[2 * tt + 1]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) us::mbar_arrive(&S.empty[slot]);
                return true;
            }
            const uint64_t* bm = reinterpret_cast<const uint64_t*>(base + (q - ch * kC) * kBm);
            const uint64_t wA = bm[lane], wB = bm[lane + 32];
            const uint32_t packed = (uint32_t)__popcll(wA) | ((uint32_t)__popcll(wB) << 16);
            uint32_t incl = packed;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += o;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t ex = incl - packed;
            const uint32_t totA = tot & 0xFFFFu;
            const bool good = S.bad[slot] == 0 && totA + (tot >> 16) <= offs[q + 1] - offs[q];
            if (!good && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
            const uint32_t* vw =
                reinterpret_cast<const uint32_t*>(base + ct * kBm + (offs[q] - offs[ch * kC]) * WB / 8u);
            const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(vw);
            // rows lane (h = 0) and lane + 32 (h = 1) step by step side by side;
            // each keeps a three-word window over its run: a step consumes at
            // most one word, and the word a step loads (predicated, only by the
            // lanes whose window moved on) is needed one step later
            uint32_t ob[2], wi[2], cur[2], nxt[2], nn[2], lo[2], hi[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint64_t w = good ? (h ? wB : wA) : 0ull;        // a bad tile decodes as zeros
                lo[h] = (uint32_t)w;
                hi[h] = (uint32_t)(w >> 32);
                ob[h] = h ? totA + (ex >> 16) : (ex & 0xFFFFu);         // element index of the row's first value
                wi[h] = ob[h] >> kLogEPW;
                cur[h] = vw[wi[h]];
                nxt[h] = vw[wi[h] + 1];
                nn[h] = vw[wi[h] + 2];
            }
            uint32_t pw[2][8];
#pragma unroll
            for (int bt = 0; bt < 8; ++bt) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t bb = __byte_perm(bt < 4 ? lo[h] : hi[h], 0u, 0x4440u | (uint32_t)(bt & 3));
                    if (bt > 0) {
                        const uint32_t nwi = ob[h] >> kLogEPW;
                        const uint32_t adv = nwi != wi[h];
                        cur[h] = adv ? nxt[h] : cur[h];
                        nxt[h] = adv ? nn[h] : nxt[h];
                        us::lds_u32_if(nn[h], adv, vbase + 4u * (nwi + 2u));
                        wi[h] = nwi;
                    }
                    // ranks ob .. ob + 7 as eight nibbles (int2: spread to sign-extended int4)
                    const uint32_t win = WB == 4 ? __funnelshift_r(cur[h], nxt[h], ob[h] << 2)
                                                 : int2x8_to_int4x8(__funnelshift_r(cur[h], nxt[h], ob[h] << 1));
                    const uint2 ent = lut[bb * kLutRep + lut_lane];
                    const uint32_t odd = win & ent.y;                       // 16 w, ranks 1,3,5,(7)
                    // 16 w, ranks 0,2,4,6; the low nibbles that the shift brings in
                    // are dropped with the odd bytes' by the pack below
                    const uint32_t even = win << 4;
                    const uint32_t d0 = __byte_perm(even, odd, ent.x);
                    const uint32_t d1 = __byte_perm(even, odd, ent.x >> 16);
                    // byte i = d0's nibble i | d1's nibble i << 4 (two's complement;
                    // the mma consumer's fp16 conversion adds the bias of 8)
                    pw[h][bt] = us::lop3<us::kLopMux>(d0 >> 4, 0x0F0F0F0Fu, d1);
                    ob[h] += ent.y & 0xFu;
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = lane + 32 * h;
                if constexpr (NT == 0) {
                    // row r: 32 bytes, its two 16-byte halves swapped on every
                    // other group of four rows (no bank conflicts either way)
                    const int sw = (r >> 2) & 1;
                    *reinterpret_cast<uint4*>(dst + r * 32 + 16 * sw) =
                        make_uint4(pw[h][0], pw[h][1], pw[h][2], pw[h][3]);
                    *reinterpret_cast<uint4*>(dst + r * 32 + 16 * (sw ^ 1)) =
                        make_uint4(pw[h][4], pw[h][5], pw[h][6], pw[h][7]);
                } else {
                    // fragment order: the 16 bytes thread (g, tig) of 16-row block
                    // mb reads are rows g and g + 8, words 2 tig and 2 tig + 1
                    const int mb = r >> 4, g = r & 7, hr = (r >> 3) & 1;
#pragma unroll
                    for (int tig = 0; tig < 4; ++tig) {
                        const int sg = mb * 32 + g * 4 + tig;
                        const int ph = sg ^ ((sg >> 3) & 3);
                        *reinterpret_cast<uint2*>(dst + ph * 16 + hr * 8) = make_uint2(pw[h][2 * tig], pw[h][2 * tig + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) us::mbar_arrive(&S.empty[slot]);
            return true;
        };

        uint8_t* dense = smem + kHeader + kLutBytes;
        bool ok = true;
        // static weights: decode this CTA's first P tiles while the previous
        // launch still runs
        for (int q = warp; q < P && ok; q += kNW) ok = decode_tile(q, dense + q * kSlot);
        // the activations are copied in by the producer warp once the previous
        // launch has finished; wait for that launch first (the wait below is
        // bounded), then for the copies
        us::pdl_wait();
        if (ok && !us::mbar_wait(&S.xfull, 0u, p.status)) {
            S.abort = 1;
            ok = false;
        }
        // the epilogue reads the row scales after the block-wide barrier
        if (p.Y && !early)
            for (int i = threadIdx.x; i < nb * kTM; i += kNW * 32) sws[i] = p.s_w[band0 * kTM + i];
        const bool all_k = p.sk_xcols == p.nTK;

        // After the wait: tile q < P is read from its dense tile; a later one is
        // decoded now into this warp's own slot (slot w held tile w, done by
        // then) and read back from there.
        int cur_b = -1;
        if constexpr (NT == 0) {
            int acc[2][N];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int n = 0; n < N; ++n) acc[h][n] = 0;
            auto flush = [&]() {
                if (cur_b < 0) return;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        atomicAdd(&accs[(cur_b * N + n) * kTM + h * 32 + lane], acc[h][n]);
                        acc[h][n] = 0;
                    }
            };
            for (int q = warp; q < per && ok; q += kNW) {
                const uint32_t ti = tinfo[q];
                const int brel = (int)(ti >> 16), tk = (int)(ti & 0x7FFFu);
                if (brel != cur_b) {
                    flush();
                    cur_b = brel;
                }
                const uint8_t* src = dense + q * kSlot;
                if (q >= P) {
                    src = dense + warp * kSlot;
                    if (!(ok = decode_tile(q, dense + warp * kSlot))) break;
                }
                // rows lane and lane + 32, eight words each: byte i of word k holds
                // positions 8k + 2i (low nibble) and 8k + 2i + 1 (high nibble), as
                // the packed activations do
                uint32_t pw[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = lane + 32 * h, sw = (r >> 2) & 1;
                    const uint4 a = *reinterpret_cast<const uint4*>(src + r * 32 + 16 * sw);
                    const uint4 b = *reinterpret_cast<const uint4*>(src + r * 32 + 16 * (sw ^ 1));
                    pw[h][0] = a.x; pw[h][1] = a.y; pw[h][2] = a.z; pw[h][3] = a.w;
                    pw[h][4] = b.x; pw[h][5] = b.y; pw[h][6] = b.z; pw[h][7] = b.w;
                }
                __syncwarp();                                 // the slot may be refilled next
                if (kSplitX && (ti & 0x8000u) && !(ok = __all_sync(0xffffffffu, us::mbar_wait(&S.xfull2, 0u, p.status)))) {
                    S.abort = 1;
                    break;
                }
                const int8_t* xt = xs + (int64_t)(all_k ? tk : q) * XROW;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
#pragma unroll
                    for (int n = 0; n < N; ++n) {
                        // even and odd positions as 16 x, against 16 w: 256 w x
                        const uint32_t xv = *reinterpret_cast<const uint32_t*>(xt + (int64_t)n * p.sk_xcols * XROW + 4 * k);
                        const int xe = (int)((xv << 4) & 0xF0F0F0F0u), xo = (int)(xv & 0xF0F0F0F0u);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            acc[h][n] = __dp4a((int)((pw[h][k] << 4) & 0xF0F0F0F0u), xe, acc[h][n]);
                            acc[h][n] = __dp4a((int)(pw[h][k] & 0xF0F0F0F0u), xo, acc[h][n]);
                        }
                    }
                }
            }
            flush();
        } else {
            // mma.sync: thread (g, tig) = (lane / 4, lane % 4) holds, for rows g
            // and g + 8 of each 16-row block, the positions 16 tig .. 16 tig + 15.
            // K is a reduction index, so it may be permuted as long as A and B
            // agree: position 16 tig + 4 kk + c is the K16 block kk's column
            // {2 tig, 2 tig + 1, 8 + 2 tig, 9 + 2 tig}[c], which makes the thread's
            // eight position pairs exactly its A fragment registers of
            // mma.m16n8k16 and its B fragment one 8-byte load per token.
            const int g = lane >> 2, tig = lane & 3;
            float acc[4][NT][4];
#pragma unroll
            for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[mb][nt][c] = 0.f;
            auto flush = [&]() {
                if (cur_b < 0) return;
#pragma unroll
                for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int row = 16 * mb + g + 8 * (c >> 1), n = 8 * nt + 2 * tig + (c & 1);
                            atomicAdd(&accs[(cur_b * NTOK + n) * kTM + row], __float2int_rn(acc[mb][nt][c]));
                            acc[mb][nt][c] = 0.f;
                        }
            };
            // word of eight two's complement nibbles w, nibbles (0,4), (1,5),
            // (2,6), (3,7) paired -> four fp16 pairs.  With u = w + 8 (the nibble
            // with its top bit flipped), 0x6400 | u is 1024 + u and 0x6400 | 16 u
            // is 1024 + 16 u: one AND and one XOR of constants, 0x6408 flipping
            // the low nibble's top bit and 0x6480 the high one's.  Then
            // (1024 + u) - 1032 and (1024 + 16 u) / 16 - 72 are w exactly
            auto cvt = [](uint32_t pw, uint32_t* o) {
                const __half2 b0 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
                const __half2 s1 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
                const __half2 b1 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));   // -72
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t v = j ? pw >> 8 : pw;
                    uint32_t l = us::lop3<us::kLopAndXor>(v, 0x000F000Fu, 0x64086408u);
                    uint32_t h = us::lop3<us::kLopAndXor>(v, 0x00F000F0u, 0x64806480u);
                    const __half2 fl = __hsub2(*reinterpret_cast<const __half2*>(&l), b0);
                    const __half2 fh = __hfma2(*reinterpret_cast<const __half2*>(&h), s1, b1);
                    o[2 * j] = *reinterpret_cast<const uint32_t*>(&fl);
                    o[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&fh);
                }
            };
            for (int q = warp; q < per && ok; q += kNW) {
                const uint32_t ti = tinfo[q];
                const int brel = (int)(ti >> 16), tk = (int)(ti & 0x7FFFu);
                if (brel != cur_b) {
                    flush();
                    cur_b = brel;
                }
                const uint8_t* src = dense + q * kSlot;
                if (q >= P) {
                    src = dense + warp * kSlot;
                    if (!(ok = decode_tile(q, dense + warp * kSlot))) break;
                }
                // B fragments: token 8 nt + g, positions 16 tig .. 16 tig + 15 as fp16
                if (kSplitX && (ti & 0x8000u) && !(ok = __all_sync(0xffffffffu, us::mbar_wait(&S.xfull2, 0u, p.status)))) {
                    S.abort = 1;
                    break;
                }
                uint32_t bf[NT][8];
                const int8_t* xt = xs + (int64_t)(all_k ? tk : q) * XROW;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 v = *reinterpret_cast<const uint2*>(xt + (int64_t)(8 * nt + g) * p.sk_xcols * XROW + 8 * tig);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t w = hh ? v.y : v.x;
                        // w + 8 per element: element 2i in byte i of lo, 2i + 1 in byte i of hi
                        const uint4 h = us::u8x8_to_f16x8(us::lop3<us::kLopAndXor>(w, 0x0F0F0F0Fu, 0x08080808u),
                                                         us::lop3<us::kLopAndXor>(w >> 4, 0x0F0F0F0Fu, 0x08080808u),
                                                         0x73625140u);
                        bf[nt][4 * hh + 0] = h.x;
                        bf[nt][4 * hh + 1] = h.y;
                        bf[nt][4 * hh + 2] = h.z;
                        bf[nt][4 * hh + 3] = h.w;
                    }
                }
                // one 16-row block at a time: its 16 bytes are loaded just before
                // they are converted, which keeps three blocks' words out of the
                // registers (4096 x 4096, N = 16: 7.50 -> 7.34 us)
#pragma unroll
                for (int mb = 0; mb < 4; ++mb) {
                    const int sg = mb * 32 + lane;
                    const uint4 av = *reinterpret_cast<const uint4*>(src + (sg ^ ((sg >> 3) & 3)) * 16);
                    uint32_t af[2][8];                        // rows g, g + 8: position pairs 0..7
                    cvt(av.x, &af[0][0]);
                    cvt(av.y, &af[0][4]);
                    cvt(av.z, &af[1][0]);
                    cvt(av.w, &af[1][4]);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            us::mma_m16n8k16_f16(acc[mb][nt], af[0][2 * kk], af[1][2 * kk], af[0][2 * kk + 1],
                                                 af[1][2 * kk + 1], bf[nt][2 * kk], bf[nt][2 * kk + 1]);
                }
                __syncwarp();                                 // the slot may be refilled next
            }
            flush();
        }
    }
    __syncthreads();
    if (S.abort && warp == kNW && lane == 0) {
        // a wait gave up: let the copies still in flight land (bounded); this
        // call's outputs are not valid (US_ERR_TIMEOUT is recorded)
        for (int ch = tail; ch < issued; ++ch) us::mbar_wait(&S.full[ch % kR], (uint32_t)(ch / kR) & 1u, nullptr);
        us::mbar_wait(&S.xfull, 0u, nullptr);
        if (S.x2) us::mbar_wait(&S.xfull2, 0u, nullptr);
    }
    us::pdl_wait();                                           // before the first global write

    // ------------------------------------------------------------- epilogue
    // dp4a accumulators hold 256 * sum (weights and activations sit in high
    // nibbles): >> 8 is exact; the mma ones hold the sum itself
    constexpr int kShift = NT ? 0 : 8;
    auto store = [&](int br, int i, int a16) {
        const int n = i / kTM, r = i - n * kTM;
        if (n >= p.N) return;                                 // padding tokens of the mma consumer
        const int m = (band0 + br) * kTM + r;
        const int a = a16 >> kShift;
        const int64_t o = (int64_t)n * p.M + m;
        p.Yacc[o] = a;
        if (p.Y) {
            const float tt = __fmul_rn(__int2float_rn(a), us::half_bits_to_float(sws[br * kTM + r]));
            p.Y[o] = us::float_to_half_bits(__fmul_rn(tt, us::half_bits_to_float(sxs[n])));
        }
    };
    // band b is owned by the CTA holding its first tile.  This CTA posts its
    // first band if that began in a lower CTA, writes the bands wholly inside
    // its range, and finishes its last band if that runs on into higher CTAs.
    uint64_t* post = reinterpret_cast<uint64_t*>(p.ws);     // G x NTOK x 64 {value, tag}
    const bool posts = band0 * p.nTK < t0;
    if (posts) {
        uint64_t* mine = post + (int64_t)cta * NTOK * kTM;
        for (int i = threadIdx.x; i < NTOK * kTM; i += kThreads)
            us::st_relaxed_gpu_u64(mine + i, (1ull << 32) | (uint32_t)accs[i]);
    }
    for (int br = posts ? 1 : 0; br < nb; ++br) {
        const int b = band0 + br;
        const int* a = accs + br * NTOK * kTM;
        if ((b + 1) * p.nTK <= t1) {                           // whole band
            for (int i = threadIdx.x; i < NTOK * kTM; i += kThreads) store(br, i, a[i]);
            continue;
        }
        // owned, continued by CTAs cta+1 .. c_hi, whose first band it is.  A
        // thread's loads of up to kE elements x 4 CTAs are all in flight before
        // the first is used, and every poll round re-loads all the words still
        // untagged together: once the last post lands, the band is seen within
        // about one L2 round trip, however many of the thread's words it held
        const int c_hi = S.c_hi;                              // b is the last band
        constexpr int kAll = NTOK * kTM;
        constexpr int kE = (kAll + kThreads - 1) / kThreads < 4 ? (kAll + kThreads - 1) / kThreads : 4;
        for (int i0 = threadIdx.x; i0 < kAll; i0 += kE * kThreads) {
            int v[kE];
#pragma unroll
            for (int e = 0; e < kE; ++e) v[e] = i0 + e * kThreads < kAll ? a[i0 + e * kThreads] : 0;
            for (int c0 = cta + 1; c0 <= c_hi; c0 += 4) {
                uint64_t w[kE][4];
                uint32_t missing = 0;                         // bit 4 e + u: word not posted yet
#pragma unroll
                for (int e = 0; e < kE; ++e)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + e * kThreads;
                        w[e][u] = c0 + u <= c_hi && i < kAll
                                      ? us::ld_relaxed_gpu_u64(post + (int64_t)(c0 + u) * kAll + i)
                                      : (1ull << 32);
                    }
#pragma unroll
                for (int e = 0; e < kE; ++e)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if ((w[e][u] >> 32) != 1ull) missing |= 1u << (4 * e + u);
                if (missing) {
                    // wait for the rest, bounded; each round polls them all at once
                    const uint64_t tw = us::globaltimer_ns();
                    while (missing) {
#pragma unroll
                        for (int e = 0; e < kE; ++e)
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                if (missing & (1u << (4 * e + u)))
                                    w[e][u] = us::ld_relaxed_gpu_u64(post + (int64_t)(c0 + u) * kAll + i0 + e * kThreads);
#pragma unroll
                        for (int e = 0; e < kE; ++e)
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                if ((w[e][u] >> 32) == 1ull) missing &= ~(1u << (4 * e + u));
                        if (missing && us::globaltimer_ns() - tw > us::kWaitLimitNs) {
                            us::set_status(p.status, US_ERR_TIMEOUT);
#pragma unroll
                            for (int e = 0; e < kE; ++e)
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    if (missing & (1u << (4 * e + u))) w[e][u] = 0;
                            break;
                        }
                    }
                }
#pragma unroll
                for (int e = 0; e < kE; ++e)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + e * kThreads;
                        if (c0 + u > c_hi || i >= kAll) continue;
                        v[e] += (int)(uint32_t)w[e][u];
                        us::st_relaxed_gpu_u64(post + (int64_t)(c0 + u) * kAll + i, 0ull);   // ready for the next call
                    }
            }
#pragma unroll
            for (int e = 0; e < kE; ++e)
                if (i0 + e * kThreads < kAll) store(br, i0 + e * kThreads, v[e]);
        }
    }
}

}  // namespace

namespace {

// Shared-memory plan of one launch; false when it does not fit.  `pre`: the
// weights are static, so tiles may be decoded before the dependency wait.
// `ie`: IE-BME super-tiles (eight run offsets per tile, their chunk bound).
struct SkPlan {
    int NT, G, per, xcols, nb, ring, slots, pre;
    size_t smem;
};

constexpr size_t kSmemTwoPerSm = 112 * 1024;   // two CTAs of this size share one SM
constexpr size_t kSmemMax = 200 * 1024;
constexpr size_t kRingMax = 64 * 1024;

#ifndef US_W4A4_DP4A_MAX_N
#define US_W4A4_DP4A_MAX_N 7         // more tokens than this: the mma.sync consumer
#endif

int nt_for_tokens(int N) { return N <= US_W4A4_DP4A_MAX_N ? 0 : (N <= 8 ? 1 : (N <= 16 ? 2 : 4)); }

bool sk_plan(int nTM, int nTK, int N, bool pre, SkPlan& pl, bool ie = false) {
    if (N < 1 || N > 32) return false;
    pl.NT = nt_for_tokens(N);
    if (pl.NT == 0 && N > 8) return false;
    if (pl.NT && nTK * kTK > (1 << 18)) return false;       // fp32 sums of int4 products stay exact
    if (!pl.NT && nTK * kTK > (1 << 17)) return false;      // int32 sums of 256 w x do not overflow
    const int ntok = ntok_for(N, pl.NT);
    const int nw = nw_for(N, pl.NT);
    const int nT = nTM * nTK;
    pl.G = us::num_sms() < nT ? us::num_sms() : nT;
    pl.per = (nT + pl.G - 1) / pl.G;
    pl.xcols = pl.per < nTK ? pl.per : nTK;
    pl.nb = (pl.per + nTK - 1) / nTK + 1;
    const size_t offs_bytes = ie ? (size_t)pl.per * 32 : (size_t)((pl.per + 1 + 3) & ~3) * 4;
    const size_t min_ring = ie ? (size_t)kMinRingIe : (size_t)kMinRing;
    const size_t fixed = kHeader + kLutBytes + offs_bytes +
                         (size_t)ntok * pl.xcols * (kTK / 2) + (size_t)pl.nb * ntok * kTM * 4 +
                         (((size_t)pl.nb * kTM + ntok) * 2 + 15) / 16 * 16 + (size_t)(pl.per * 4 + 15) / 16 * 16;
    // every warp needs a slot of its own; static weights want one per tile
    const int want = pre ? (pl.per > nw ? pl.per : nw) : nw;
    for (size_t budget : {kSmemTwoPerSm, kSmemMax}) {
        if (fixed + min_ring + (size_t)nw * kSlot > budget) continue;
        const size_t cap = (budget - fixed - min_ring) / kSlot;
        pl.slots = (int)((size_t)want < cap ? (size_t)want : cap);
        pl.pre = pre ? (pl.per < pl.slots ? pl.per : pl.slots) : 0;
        size_t ring = budget - fixed - (size_t)pl.slots * kSlot;
        if (ring > kRingMax) ring = kRingMax;
        ring &= ~(size_t)15;
        pl.ring = (int)ring;
        pl.smem = fixed + (size_t)pl.slots * kSlot + ring;
        return true;
    }
    return false;
}

template <int N, int NT, bool IE = false>
us_status launch_sk_n(UsKParams p, const SkPlan& pl, cudaStream_t st) {
    void (*kern)(UsKParams);
    if constexpr (IE)
        kern = w4a4_sk_kernel<N, NT, 4, true>;
    else
        kern = p.elem == US_I2 ? w4a4_sk_kernel<N, NT, 2> : w4a4_sk_kernel<N, NT, 4>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return US_ERR_CUDA;
    p.sk_grid = pl.G; p.sk_per = pl.per; p.sk_ring = pl.ring; p.sk_xcols = pl.xcols; p.sk_nb = pl.nb;
    p.sk_slots = pl.slots; p.sk_pre = pl.pre;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.G);
    cfg.blockDim = dim3(threads_for(N, NT));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace
