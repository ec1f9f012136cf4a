// us_w4a4_sk.cu -- W4A4 bitmap SpMM for 1..8 tokens, the tile sequence spread
// evenly over the SMs.
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
//    1-D bulk copies (TMA).  Every chunk is requested as soon as there is room:
//    the runs are packed into a byte ring by their real length, not their worst
//    case, so at 50 % density about twice as many tiles are in flight;
//  * work item = one tile on one warp; lane l decodes rows l and l+32.  Row
//    bases come from one warp scan of packed popcounts (the word-level part of
//    UnionSparse's idx_base, section VI-B);
//  * byte-step decode as in the cluster kernel (selector table + PRMT, dp4a on
//    16*w); each table entry also carries the mask that empties rank 7's byte
//    (clear positions read it) unless all eight positions are set;
//  * a band split between CTAs is finished by the CTA holding its first tile:
//    the others post their partial sums as 64-bit {value, tag} words (one
//    relaxed store each, no fence, no counter: the tag arrives with its value)
//    and the owner waits for the tags (bounded), adds, and clears them for the
//    next call.  Partials are integers, so the sum is exact in any order;
//  * programmatic stream serialisation: barrier and table set-up (and, for
//    weights flagged static, the weight copies) overlap the previous launch.
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
    return NT ? (NT == 1 ? 12 : (NT == 2 ? 8 : 6)) : (N == 1 ? 16 : (N <= 3 ? 12 : 8));
}
__host__ __device__ constexpr int threads_for(int N, int NT) { return (nw_for(N, NT) + 1) * 32; }
__host__ __device__ constexpr int ntok_for(int N, int NT) { return NT ? 8 * NT : N; }   // token slots
__host__ __device__ constexpr int xrow_for(int NT) { return NT ? 32 : 64; }            // staged bytes per K tile
constexpr int kLutRep = 16;                 // selector table replicas (bank spreading)
constexpr int kHeader = 512;
constexpr int kLutBytes = 256 * kLutRep * 8;   // {selector pair, odd-rank mask} per entry
constexpr int kMinRing = 3 * kC * (kBm + kValCap);   // at least three worst-case chunks

struct SkSmem {
    uint64_t full[kR], empty[kR];
    uint32_t pos[kR];                       // ring offset of the chunk in slot s
    uint32_t bad[kR];                       // its offsets failed the checks
    uint32_t abort;
};
static_assert(sizeof(SkSmem) <= kHeader, "header");

__host__ __device__ inline int sk_cta_of(int64_t t, int G, int nT) { return (int)(((t + 1) * G - 1) / nT); }
__host__ __device__ inline int sk_start(int c, int G, int nT) { return (int)((int64_t)c * nT / G); }


template <int N, int NT>
__global__ void __launch_bounds__(threads_for(N, NT), 2)   // two per SM: this launch and the next
w4a4_sk_kernel(const UsKParams p) {
    constexpr int kNW = nw_for(N, NT);
    constexpr int kThreads = threads_for(N, NT);
    constexpr int NTOK = ntok_for(N, NT);
    constexpr int XROW = xrow_for(NT);
    extern __shared__ __align__(128) uint8_t smem[];
    SkSmem& S = *reinterpret_cast<SkSmem*>(smem);
    uint2* lut = reinterpret_cast<uint2*>(smem + kHeader);
    uint8_t* ring = smem + kHeader + kLutBytes;
    const uint32_t D = (uint32_t)p.sk_ring;
    const int nT = p.nTM * p.nTK, G = p.sk_grid;
    const int cta = blockIdx.x;
    const int t0 = sk_start(cta, G, nT), t1 = sk_start(cta + 1, G, nT);
    const int per = t1 - t0;
    uint32_t* offs = reinterpret_cast<uint32_t*>(ring + D);                       // per + 1
    // activations: NTOK x xcols x XROW bytes (int8 per position for dp4a, the
    // packed int4 codes for mma)
    int8_t* xs = reinterpret_cast<int8_t*>(offs + ((p.sk_per + 1 + 3) & ~3));
    int* accs = reinterpret_cast<int*>(xs + NTOK * p.sk_xcols * XROW);           // bands x NTOK x 64
    uint16_t* sws = reinterpret_cast<uint16_t*>(accs + p.sk_nb * NTOK * kTM);     // bands x 64 row scales
    uint16_t* sxs = sws + p.sk_nb * kTM;                                          // NTOK token scales
    const int band0 = t0 / p.nTK;
    const int nb = (t1 - 1) / p.nTK - band0 + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool early = (p.flags & US_BITMAP_STATIC) != 0;   // weights may be fetched before the wait

    if (threadIdx.x == 0) {
        for (int i = 0; i < kR; ++i) {
            us::mbar_init(&S.full[i], 1);
            us::mbar_init(&S.empty[i], kC);                  // one arrival per tile
        }
        S.abort = 0;
        us::fence_mbar_init();
    }
    for (int i = threadIdx.x; i < nb * NTOK * kTM; i += kThreads) accs[i] = 0;
    __syncthreads();
    us::pdl_launch_dependents();

    int issued = 0, tail = 0;                                 // producer bookkeeping (lane 0)
    if (warp == kNW) {
        // ------------------------------------------------------------ producer
        if (!early) us::pdl_wait();
        for (int i = lane; i <= per; i += 32) offs[i] = p.tile_off[t0 + i];
        __syncwarp();
        const int nch = (per + kC - 1) / kC;
        uint32_t pos = 0;                                     // end of the newest chunk in the ring
        bool waited = !early;
        for (int ch = 0; ch < nch; ++ch) {
            const int q0 = ch * kC, ct = min(kC, per - q0), slot = ch % kR;
            bool ok = true;
            if (lane < ct) {
                const uint32_t a = offs[q0 + lane], e = offs[q0 + lane + 1];
                ok = e >= a && (e - a) <= (uint32_t)(kTM * kTK) && (a & 31u) == 0 && (e & 31u) == 0 &&
                     (uint64_t)e * 4u <= p.values_bytes * 8ull;
            }
            const bool all_ok = __all_sync(0xffffffffu, ok);
            int fail = 0;
            if (lane == 0) {
                const uint32_t vb = all_ok ? (offs[q0 + ct] - offs[q0]) / 2u : 0u;
                const uint32_t sz = (uint32_t)ct * kBm + vb;
                // room for sz bytes: the ring holds the chunks [tail, ch) in order,
                // from the start of chunk `tail` to `pos`, wrapping at D
                uint32_t place = 0;
                for (;;) {
                    const int inflight = ch - tail;
                    if (inflight == 0) { place = 0; break; }
                    if (inflight < kR) {
                        const uint32_t s0 = S.pos[tail % kR];
                        if (pos > s0) {
                            if (pos + sz <= D) { place = pos; break; }
                            if (sz <= s0) { place = 0; break; }
                        } else if (pos + sz <= s0) {
                            place = pos;
                            break;
                        }
                    }
                    // the consumers start only after the previous launch has finished:
                    // wait for that too before a bounded wait on them
                    if (!waited) {
                        us::pdl_wait();
                        waited = true;
                    }
                    if (!us::mbar_wait(&S.empty[tail % kR], (uint32_t)(tail / kR) & 1u, p.status)) {
                        fail = 1;
                        break;
                    }
                    ++tail;
                }
                if (!fail) {
                    if (!all_ok) us::set_status(p.status, US_ERR_CORRUPT);
                    S.pos[slot] = place;
                    S.bad[slot] = all_ok ? 0u : 1u;
                    us::mbar_arrive_expect_tx(&S.full[slot], sz);
                    us::bulk_g2s(ring + place, p.bitmap + (int64_t)(t0 + q0) * (kBm / 8), (uint32_t)ct * kBm,
                                 &S.full[slot]);
                    if (vb) us::bulk_g2s(ring + place + ct * kBm, p.values + offs[q0] / 2u, vb, &S.full[slot]);
                    // a short last chunk has fewer tiles: arrive for the missing ones
                    for (int i = ct; i < kC; ++i) us::mbar_arrive(&S.empty[slot]);
                    pos = place + sz;
                    issued = ch + 1;
                }
            }
            if (__shfl_sync(0xffffffffu, fail, 0)) {
                S.abort = 1;
                break;
            }
        }
        if (!waited) us::pdl_wait();                          // idle now: take it off the epilogue's path
    }
    else {
        // ----------------------------------------------------------- consumers
        for (int e = threadIdx.x; e < 256; e += kNW * 32) {
            // clear positions take rank 7's byte, which must then be empty (dp4a:
            // 16 w = 0; mma: w + 8 = 8): the odd-rank mask drops rank 7 unless all
            // eight positions are set
            const uint32_t full = NT ? 0x0F0F0F0Fu : 0xF0F0F0F0u, part = NT ? 0x000F0F0Fu : 0x00F0F0F0u;
            const uint2 ent = make_uint2(us::make_sel((uint32_t)e), e == 255 ? full : part);
#pragma unroll
            for (int r = 0; r < kLutRep; ++r) lut[e * kLutRep + r] = ent;
        }
        us::pdl_wait();
        // activations: column block xq of token n holds K tile tk, where xq = tk when
        // the CTA spans a whole band width, else xq = the tile's place in the range
        {
            const uint8_t* xg = reinterpret_cast<const uint8_t*>(p.X);
            const int xcols = p.sk_xcols;
            const bool all_k = xcols == p.nTK;
            const int tk0 = t0 % p.nTK;
            const int ncols = all_k ? p.nTK : per;
            // every load of a round is issued before its stores (the first global
            // round trip after the dependency wait is on the critical path).
            // dp4a: 4-byte words (8 codes, 8 per K tile) spread over many
            // threads, each expanded to 8 int8; mma: 16-byte pieces (32 codes, 2
            // per K tile) copied as they are
            constexpr int kPieceB = NT ? 16 : 4;
            constexpr int kPerTile = 32 / kPieceB;
            const int pieces = ncols * kPerTile;
            const int total = NTOK * pieces;
            constexpr int kU = (NT == 1 || NT == 2) ? 8 : 4;
            for (int i0 = threadIdx.x; i0 < total; i0 += kU * kNW * 32) {
                uint4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = i0 + u * kNW * 32;
                    v[u] = make_uint4(0u, 0u, 0u, 0u);              // absent tokens: code 0
                    if (i < total) {
                        const int n = i / pieces, r = i - n * pieces, xq = r / kPerTile, hh = r - xq * kPerTile;
                        const int tk = all_k ? xq : (tk0 + xq) % p.nTK;
                        const uint8_t* src = xg + (int64_t)n * (p.K / 2) + (int64_t)tk * (kTK / 2) + kPieceB * hh;
                        if (n < p.N) {
                            if (NT) v[u] = __ldg(reinterpret_cast<const uint4*>(src));
                            else v[u].x = __ldg(reinterpret_cast<const uint32_t*>(src));
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = i0 + u * kNW * 32;
                    if (i >= total) break;
                    const int n = i / pieces, r = i - n * pieces, xq = r / kPerTile, hh = r - xq * kPerTile;
                    if (NT) {
                        *reinterpret_cast<uint4*>(xs + ((int64_t)n * xcols + xq) * XROW + 16 * hh) = v[u];
                    } else {
                        const uint32_t lo = v[u].x & 0x0F0F0F0Fu, hi = (v[u].x >> 4) & 0x0F0F0F0Fu;
                        const uint32_t e0 = __vsub4(__byte_perm(lo, hi, 0x5140) ^ 0x08080808u, 0x08080808u);
                        const uint32_t e1 = __vsub4(__byte_perm(lo, hi, 0x7362) ^ 0x08080808u, 0x08080808u);
                        *reinterpret_cast<uint2*>(xs + ((int64_t)n * xcols + xq) * XROW + 8 * hh) = make_uint2(e0, e1);
                    }
                }
            }
        }
        if (p.Y) {
            for (int i = threadIdx.x; i < nb * kTM; i += kNW * 32) sws[i] = p.s_w[band0 * kTM + i];
            for (int i = threadIdx.x; i < NTOK; i += kNW * 32) sxs[i] = i < p.N ? p.s_x[i] : (uint16_t)0;
        }
        us::named_bar_sync(1, kNW * 32);

        if constexpr (NT == 0) {
            const uint32_t lut_lane = (uint32_t)(lane % kLutRep);
            const bool all_k = p.sk_xcols == p.nTK;
            int acc[2][N];
    #pragma unroll
            for (int h = 0; h < 2; ++h)
    #pragma unroll
                for (int n = 0; n < N; ++n) acc[h][n] = 0;
            int cur_b = -1;
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
            // one tile per warp at a time; lane l decodes rows l and l + 32
            for (int q = warp; q < per; q += kNW) {
                const int ch = q / kC, slot = ch % kR;
                if (!us::mbar_wait(&S.full[slot], (uint32_t)(ch / kR) & 1u, p.status)) {
                    S.abort = 1;
                    break;
                }
                const int t = t0 + q;
                const int brel = t / p.nTK - band0;
                if (brel != cur_b) {
                    flush();
                    cur_b = brel;
                }
                const int ct = min(kC, per - ch * kC);
                const uint8_t* base = ring + S.pos[slot];
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
                if (!good) {
                    if (lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
                } else {
                    const uint32_t* vw = reinterpret_cast<const uint32_t*>(base + ct * kBm + (offs[q] - offs[ch * kC]) / 2u);
                    const int8_t* xt = xs + (all_k ? t % p.nTK : q) * kTK;
                    const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(vw);
    #pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t w = h ? wB : wA;
                        const uint32_t lo = (uint32_t)w, hi = (uint32_t)(w >> 32);
                        uint32_t ob = h ? totA + (ex >> 16) : (ex & 0xFFFFu);   // nibble index of the row's first value
                        // two-word window over the row's run; a step consumes at most one
                        // word, so a new word is loaded only by the lanes whose window
                        // moved on (predicated, no branch): fewer bank conflicts
                        uint32_t wi = ob >> 3;
                        uint32_t cur = vw[wi], nxt = vw[wi + 1];
    #pragma unroll
                        for (int bt = 0; bt < 8; ++bt) {
                            const uint32_t bb = __byte_perm(bt < 4 ? lo : hi, 0u, 0x4440u | (uint32_t)(bt & 3));
                            if (bt > 0) {
                                const uint32_t nwi = ob >> 3;
                                const uint32_t adv = nwi != wi;
                                cur = adv ? nxt : cur;
                                us::lds_u32_if(nxt, adv, vbase + 4u * (nwi + 1u));
                                wi = nwi;
                            }
                            const uint32_t win = __funnelshift_r(cur, nxt, ob << 2);
                            const uint2 ent = lut[bb * kLutRep + lut_lane];
                            const uint32_t odd = win & ent.y;                       // 16 w, ranks 1,3,5,(7)
                            const uint32_t even = (win << 4) & 0xF0F0F0F0u;         // 16 w, ranks 0,2,4,6
                            const int d0 = (int)__byte_perm(even, odd, ent.x);
                            const int d1 = (int)__byte_perm(even, odd, ent.x >> 16);
    #pragma unroll
                            for (int n = 0; n < N; ++n) {
                                const uint2 xv =
                                    *reinterpret_cast<const uint2*>(xt + (int64_t)n * p.sk_xcols * kTK + 8 * bt);
                                acc[h][n] = __dp4a(d0, (int)xv.x, acc[h][n]);
                                acc[h][n] = __dp4a(d1, (int)xv.y, acc[h][n]);
                            }
                            ob += (uint32_t)__popc(bb);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) us::mbar_arrive(&S.empty[slot]);
            }
            flush();
        } else {
            // mma.sync consumer: one tile per warp at a time.  Thread (g, tig) =
            // (lane / 4, lane % 4) decodes, for rows g and g + 8 of each 16-row
            // block, the 16 consecutive positions 16 tig .. 16 tig + 15 (two
            // byte-steps) as fp16.  K is a reduction index, so it may be permuted
            // as long as A and B agree: position 16 tig + 4 kk + c is the K16 block
            // kk's column {2 tig, 2 tig + 1, 8 + 2 tig, 9 + 2 tig}[c], which makes the
            // decoded halves exactly the thread's A fragment registers of
            // mma.m16n8k16 and its B fragment one 8-byte load per token.
            const int g = lane >> 2, tig = lane & 3;
            const uint32_t lut_lane = (uint32_t)(lane % kLutRep);
            const bool all_k = p.sk_xcols == p.nTK;
            const uint32_t m_lo = tig == 0 ? 0u : (tig == 1 ? 0xFFFFu : 0xFFFFFFFFu);   // bits below 16 tig
            const uint32_t m_hi = tig == 3 ? 0xFFFFu : 0u;
            const uint32_t sh16 = 16u * (uint32_t)(tig & 1);
            float acc[4][NT][4];
#pragma unroll
            for (int mb = 0; mb < 4; ++mb)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[mb][nt][c] = 0.f;
            int cur_b = -1;
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
            for (int q = warp; q < per; q += kNW) {
                const int ch = q / kC, slot = ch % kR;
                if (!us::mbar_wait(&S.full[slot], (uint32_t)(ch / kR) & 1u, p.status)) {
                    S.abort = 1;
                    break;
                }
                const int t = t0 + q;
                const int brel = t / p.nTK - band0;
                if (brel != cur_b) {
                    flush();
                    cur_b = brel;
                }
                const int ct = min(kC, per - ch * kC);
                const uint8_t* base = ring + S.pos[slot];
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
                if (!good) {
                    if (lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
                } else {
                    const uint32_t* vw = reinterpret_cast<const uint32_t*>(base + ct * kBm + (offs[q] - offs[ch * kC]) / 2u);
                    const uint32_t vbase = (uint32_t)__cvta_generic_to_shared(vw);
                    // B fragments: token 8 nt + g, positions 16 tig .. 16 tig + 15 as fp16
                    uint32_t bf[NT][8];
                    const int xq = all_k ? t % p.nTK : q;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint2 v = *reinterpret_cast<const uint2*>(
                            xs + ((int64_t)(8 * nt + g) * p.sk_xcols + xq) * XROW + 8 * tig);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint32_t w = hh ? v.y : v.x;
                            // w + 8 per element: element 2i in byte i of lo, 2i + 1 in byte i of hi
                            const uint4 h = us::u8x8_to_f16x8((w & 0x0F0F0F0Fu) ^ 0x08080808u,
                                                             ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u, 0x73625140u);
                            bf[nt][4 * hh + 0] = h.x;
                            bf[nt][4 * hh + 1] = h.y;
                            bf[nt][4 * hh + 2] = h.z;
                            bf[nt][4 * hh + 3] = h.w;
                        }
                    }
#pragma unroll
                    for (int mb = 0; mb < 4; ++mb) {
                        uint32_t af[2][8];                        // rows g, g + 8: 16 positions as fp16 pairs
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int r = 16 * mb + g + 8 * hr;
                            const uint64_t word = bm[r];
                            const uint32_t e = __shfl_sync(0xffffffffu, ex, r & 31);
                            const uint32_t rowbase = r < 32 ? (e & 0xFFFFu) : totA + (e >> 16);
                            const uint32_t lo = (uint32_t)word, hi = (uint32_t)(word >> 32);
                            const uint32_t w16 = ((tig < 2 ? lo : hi) >> sh16) & 0xFFFFu;
                            uint32_t ob = rowbase + (uint32_t)__popc(lo & m_lo) + (uint32_t)__popc(hi & m_hi);
                            uint32_t wi = ob >> 3;
                            uint32_t cur = vw[wi], nxt = vw[wi + 1];
#pragma unroll
                            for (int s2 = 0; s2 < 2; ++s2) {
                                const uint32_t bb = s2 ? (w16 >> 8) : (w16 & 0xFFu);
                                if (s2) {
                                    const uint32_t nwi = ob >> 3;
                                    const uint32_t adv = nwi != wi;
                                    cur = adv ? nxt : cur;
                                    us::lds_u32_if(nxt, adv, vbase + 4u * (nwi + 1u));
                                    wi = nwi;
                                }
                                const uint32_t win = __funnelshift_r(cur, nxt, ob << 2);
                                const uint2 ent = lut[bb * kLutRep + lut_lane];
                                const uint32_t even = (win & 0x0F0F0F0Fu) ^ 0x08080808u;        // w + 8, ranks 0,2,4,6
                                const uint32_t odd = ((win >> 4) & ent.y) ^ 0x08080808u;        // w + 8, ranks 1,3,5,(7)
                                const uint4 h = us::u8x8_to_f16x8(even, odd, ent.x);
                                af[hr][4 * s2 + 0] = h.x;
                                af[hr][4 * s2 + 1] = h.y;
                                af[hr][4 * s2 + 2] = h.z;
                                af[hr][4 * s2 + 3] = h.w;
                                ob += (uint32_t)__popc(bb);
                            }
                        }
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                us::mma_m16n8k16_f16(acc[mb][nt], af[0][2 * kk], af[1][2 * kk], af[0][2 * kk + 1],
                                                     af[1][2 * kk + 1], bf[nt][2 * kk], bf[nt][2 * kk + 1]);
                    }
                }
                __syncwarp();
                if (lane == 0) us::mbar_arrive(&S.empty[slot]);
            }
            flush();
        }
    }
    __syncthreads();
    if (S.abort && warp == kNW && lane == 0) {
        // a wait gave up: let the copies still in flight land (bounded); this
        // call's outputs are not valid (US_ERR_TIMEOUT is recorded)
        for (int ch = tail; ch < issued; ++ch) us::mbar_wait(&S.full[ch % kR], (uint32_t)(ch / kR) & 1u, nullptr);
    }
    us::pdl_wait();                                           // before the first global write

    // ------------------------------------------------------------- epilogue
    // dp4a accumulators hold 16 * sum (weights sit in the high nibble): >> 4 is
    // exact; the mma ones hold the sum itself
    constexpr int kShift = NT ? 0 : 4;
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
        // owned, continued by CTAs cta+1 .. c_hi, whose first band it is
        const int c_hi = sk_cta_of((int64_t)(b + 1) * p.nTK - 1, G, nT);
        for (int i = threadIdx.x; i < NTOK * kTM; i += kThreads) {
            int v = a[i];
            for (int c0 = cta + 1; c0 <= c_hi; c0 += 4) {
                uint64_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    w[u] = c0 + u <= c_hi ? us::ld_relaxed_gpu_u64(post + (int64_t)(c0 + u) * NTOK * kTM + i)
                                          : (1ull << 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (c0 + u > c_hi) continue;
                    uint64_t* src = post + (int64_t)(c0 + u) * NTOK * kTM + i;
                    if ((w[u] >> 32) != 1ull) {
                        // not posted yet: wait for it, bounded
                        const uint64_t tw = us::globaltimer_ns();
                        while (((w[u] = us::ld_relaxed_gpu_u64(src)) >> 32) != 1ull) {
                            if (us::globaltimer_ns() - tw > us::kWaitLimitNs) {
                                us::set_status(p.status, US_ERR_TIMEOUT);
                                w[u] = 0;
                                break;
                            }
                        }
                    }
                    v += (int)(uint32_t)w[u];
                    us::st_relaxed_gpu_u64(src, 0ull);               // ready for the next call
                }
            }
            store(br, i, v);
        }
    }
}

}  // namespace

namespace {

// Shared-memory plan of one launch; false when it does not fit.
struct SkPlan {
    int NT, G, per, xcols, nb, ring;
    size_t smem;
};

constexpr size_t kSmemTwoPerSm = 112 * 1024;   // two CTAs of this size share one SM
constexpr size_t kSmemMax = 200 * 1024;

#ifndef US_W4A4_DP4A_MAX_N
#define US_W4A4_DP4A_MAX_N 7         // more tokens than this: the mma.sync consumer
#endif

int nt_for_tokens(int N) { return N <= US_W4A4_DP4A_MAX_N ? 0 : (N <= 8 ? 1 : (N <= 16 ? 2 : 4)); }

bool sk_plan(int nTM, int nTK, int N, SkPlan& pl) {
    if (N < 1 || N > 32) return false;
    pl.NT = nt_for_tokens(N);
    if (pl.NT == 0 && N > 8) return false;
    if (pl.NT && nTK * kTK > (1 << 18)) return false;       // fp32 sums of int4 products stay exact
    const int ntok = ntok_for(N, pl.NT), xrow = xrow_for(pl.NT);
    const int nT = nTM * nTK;
    pl.G = us::num_sms() < nT ? us::num_sms() : nT;
    pl.per = (nT + pl.G - 1) / pl.G;
    pl.xcols = pl.per < nTK ? pl.per : nTK;
    pl.nb = (pl.per + nTK - 1) / nTK + 1;
    const size_t fixed = kHeader + kLutBytes + (size_t)((pl.per + 1 + 3) & ~3) * 4 +
                         (size_t)ntok * pl.xcols * xrow + (size_t)pl.nb * ntok * kTM * 4 +
                         (((size_t)pl.nb * kTM + ntok) * 2 + 15) / 16 * 16;
    const size_t ring_max = 64 * 1024;
    size_t ring = fixed < kSmemTwoPerSm ? kSmemTwoPerSm - fixed : 0;
    if (ring < kMinRing) ring = fixed < kSmemMax ? kSmemMax - fixed : 0;   // then one CTA per SM
    if (ring > ring_max) ring = ring_max;
    ring &= ~(size_t)15;
    if (ring < kMinRing) return false;
    pl.ring = (int)ring;
    pl.smem = fixed + ring;
    return pl.smem <= kSmemMax;
}

template <int N, int NT>
us_status launch_sk_n(UsKParams p, const SkPlan& pl, cudaStream_t st) {
    auto kern = w4a4_sk_kernel<N, NT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return US_ERR_CUDA;
    p.sk_grid = pl.G; p.sk_per = pl.per; p.sk_ring = pl.ring; p.sk_xcols = pl.xcols; p.sk_nb = pl.nb;
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

namespace us {

bool w4a4_sk_supported(int TM, int TK, int M, int K, int N) {
    if (TM != kTM || TK != kTK) return false;
    SkPlan pl;
    return sk_plan(M / TM, K / TK, N, pl);
}

size_t w4a4_sk_ws(int M, int K, int N) {
    SkPlan pl;
    if (!sk_plan(M / kTM, K / kTK, N, pl)) return 0;
    return (size_t)pl.G * ntok_for(N, pl.NT) * kTM * 8;   // one posted partial per CTA
}

int w4a4_sk_variant(int N) { return nt_for_tokens(N); }

// p.ws: the workspace, G x NTOK x 64 posted {value, tag} words, zero before the
// first call and left zero by every call.
us_status launch_w4a4_sk(UsKParams p, cudaStream_t st) {
    SkPlan pl;
    if (!sk_plan(p.nTM, p.nTK, p.N, pl)) return US_ERR_UNSUPPORTED;
    switch (pl.NT) {
        case 1: return launch_sk_n<8, 1>(p, pl, st);
        case 2: return launch_sk_n<16, 2>(p, pl, st);
        case 4: return launch_sk_n<32, 4>(p, pl, st);
        default: break;
    }
    switch (p.N) {
        case 1: return launch_sk_n<1, 0>(p, pl, st);
        case 2: return launch_sk_n<2, 0>(p, pl, st);
        case 3: return launch_sk_n<3, 0>(p, pl, st);
        case 4: return launch_sk_n<4, 0>(p, pl, st);
        case 5: return launch_sk_n<5, 0>(p, pl, st);
        case 6: return launch_sk_n<6, 0>(p, pl, st);
        case 7: return launch_sk_n<7, 0>(p, pl, st);
        case 8: return launch_sk_n<8, 0>(p, pl, st);
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
