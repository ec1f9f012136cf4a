// us_spmspv_stream.cu -- fp16 spMspV on 64 x 64 column-scan tiles, streamed.
//
// y = (W (.) M) . (x (.) M(x)): static bitmap sparsity of W and the dynamic
// mask that keeps column k iff |x_k| > tau ("Unified Static-Dynamic Pruning
// for Efficient LLM Inference", section 2 and section 4.2).  W is stored
// column-major inside its tiles (Tiled-CBC scan, same page section 4.1), so the
// nonzeros of one tile column are one contiguous run.
//
// A tile's bitmap (512 B) and its whole value run are one contiguous piece of
// each array, and so are those of consecutive tiles of a band.  Gathering only
// the active columns' runs (about 64 B each at 50 % weight density) moves
// fewer bytes but at sector granularity and one round trip per column; here
// the runs are streamed instead, and the selection happens in shared memory:
//  * per CTA one tile-row band x one K slice (the slices of a band form one
//    thread-block cluster; slices are chosen so that three CTAs share each SM
//    evenly); a producer lane copies chunks of two consecutive tiles - their
//    bitmaps and their value runs, two 1-D bulk copies (TMA) - into a byte
//    ring, placed by real length (the asynchronous metadata-then-data pipeline
//    of SPDP section 4.2.2, with the whole tile as the unit).  Measured on
//    14336 x 4096: an L2 bulk prefetch of each CTA's range ahead of the ring
//    made the stream slower (18.3 against 14.6 us with the consumers' work
//    left out), and so did chunks of four tiles (19.6 us);
//  * a consumer warp takes a whole tile: column popcounts and a warp scan give
//    each column's base in the run; a ballot of "popcount > 0 and
//    |x_j| > tau" lists the active columns and compacts them;
//  * sixteen active columns at a time, the lanes copy the columns' nonzeros
//    into a zero-filled strip that holds the compacted columns column-major
//    (64 rows per column, 16-byte chunks XOR-swizzled by column): set bit i of
//    the column word is row i, its value the next one of the column's run -
//    the base-plus-rank addressing of HAD-SMBD.  Two lanes share a column
//    (rows 0-31 and 32-63), four when the group has at most eight columns
//    (each half-word split at its middle set bit, one lane walking up from
//    the first, one down from the last); the ring slot is released once the
//    tile's last column is copied;
//  * ldmatrix.trans turns the strip into m16n8k16 A fragments and mma.sync
//    multiplies them with the compacted activations, fp32 accumulation;
//  * warp partials are summed in fixed warp order and the K slices of a band
//    in fixed rank order through distributed shared memory: repeated calls
//    are bitwise identical.
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kTM = 64, kTK = 64;
constexpr int kBm = kTM * kTK / 8;           // bitmap bytes per tile
constexpr int kValCap = kTM * kTK * 2;       // value bytes per tile, worst case
constexpr int kC = 2;                        // tiles per chunk
constexpr int kR = 16;                       // chunks in flight at most (mbarrier pairs)
constexpr int kNW = 6;                       // consumer warps
constexpr int kThreads = (kNW + 1) * 32;     // + the producer warp
constexpr int kHeader = 512;
constexpr int kMaxNk = 128;                  // K tiles per slice (staged activations)
constexpr int kGroup = 16;                   // compacted columns per pass
constexpr int kStrip = kGroup * 128;         // kGroup columns x 64 rows of fp16
constexpr int kTable = 64 * 16;              // per active column: word, bases, x
constexpr int kWarpBytes = kStrip + kTable + 128;
constexpr int kMinRing = 2 * kC * (kBm + kValCap);

struct SvSmem {
    uint64_t full[kR], empty[kR];
    uint64_t xfull;
    uint32_t pos[kR];
    uint32_t bad[kR];
    uint32_t abort;
};
static_assert(sizeof(SvSmem) <= kHeader, "header");

struct ColEnt {                               // one active column of a tile
    uint32_t lo, hi;                          // column word: bit i = row i
    uint32_t base;                            // first value of the column in the tile's run
    uint32_t x;                               // fp16 activation (low 16 bits), popc(lo) << 16
};

US_DEV void ldsm_x4_trans(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}

// Copies `cnt` of the set bits of the 32-bit column segment w into the strip
// column col: walking up from the lowest set bit (down = 0, values run[r],
// run[r + 1], ...) or down from the highest (down = 1, values run[r],
// run[r - 1], ...).  Bit i is row (r0 / 2) + i, stored at byte (r0 | 2 i) ^ sw
// of the column.
US_DEV uint16_t lds_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
US_DEV void sts_u16(uint32_t addr, uint16_t v) { asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v)); }

// (shared-memory addresses: src = the value of the first bit walked, colk =
// the strip column's address with its half-word offset and swizzle folded in:
// row bit i lands at colk ^ 2 i, since 2 i only touches bits 1-5)
US_DEV uint32_t flo(uint32_t w) {
    uint32_t r;
    asm("bfind.u32 %0, %1;" : "=r"(r) : "r"(w));
    return r;
}
US_DEV void scatter_half(uint32_t w, uint32_t cnt, int down, uint32_t src, uint32_t colk) {
    if (!down) {
        for (uint32_t k = 0; k < cnt; ++k, src += 2u) {
            const uint32_t i = (uint32_t)__ffs(w) - 1u;
            w &= w - 1u;
            sts_u16(colk ^ (2u * i), lds_u16(src));
        }
    } else {
        // two bits per round, the second one predicated
        for (uint32_t k = 0; k < cnt; k += 2u, src -= 4u) {
            const uint32_t i0 = flo(w);
            w ^= 1u << i0;
            const uint16_t v0 = lds_u16(src);
            sts_u16(colk ^ (2u * i0), v0);
            if (k + 1u < cnt) {
                const uint32_t i1 = flo(w);
                w ^= 1u << i1;
                sts_u16(colk ^ (2u * i1), lds_u16(src - 2u));
            }
        }
    }
}

// smem layout offsets (identical in every CTA of a cluster: the reduction
// reads the other CTAs' partials at this CTA's offset)
struct SvLayout {
    uint32_t offs, xs, warps, red, ring;
};
__host__ __device__ inline SvLayout sv_layout(int nk_max) {
    SvLayout L;
    L.offs = kHeader;
    L.xs = L.offs + (((uint32_t)nk_max + 1u) * 4u + 15u) / 16u * 16u;
    L.warps = L.xs + (uint32_t)nk_max * kTK * 2u;
    L.warps = (L.warps + 127u) & ~127u;
    L.red = L.warps + (uint32_t)kNW * kWarpBytes;
    L.ring = L.red + (uint32_t)(kNW + 1) * kTM * 4u;
    return L;
}

__global__ void __launch_bounds__(kThreads, 3)
spmspv_stream_kernel(const UsKParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    SvSmem& S = *reinterpret_cast<SvSmem*>(smem);
    const int band = blockIdx.x / p.split;           // the split slices of a band form one cluster
    const int slice = blockIdx.x % p.split;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int nk_max = (p.nTK + p.split - 1) / p.split;
    const SvLayout L = sv_layout(nk_max);
    uint32_t* offs = reinterpret_cast<uint32_t*>(smem + L.offs);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    uint8_t* ring = smem + L.ring;
    const uint32_t D = (uint32_t)p.sk_ring;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool early = (p.flags & US_BITMAP_STATIC) != 0;
    const int64_t tile0 = (int64_t)band * p.nTK + kt0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kR; ++i) {
            us::mbar_init(&S.full[i], 1);
            us::mbar_init(&S.empty[i], kC);                // one arrival per tile
        }
        us::mbar_init(&S.xfull, 1);
        S.abort = 0;
        us::fence_mbar_init();
    }
    __syncthreads();
    us::pdl_launch_dependents();

    int issued = 0, tail = 0;                              // producer bookkeeping (lane 0)
    float acc[4][4];
#pragma unroll
    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[mb][c] = 0.f;

    if (warp == kNW) {
        // ------------------------------------------------------------ producer
        if (!early) us::pdl_wait();
        for (int i = lane; i <= nk; i += 32) offs[i] = p.tile_off[tile0 + i];
        __syncwarp();
        const int nch = (nk + kC - 1) / kC;
        uint32_t pos = 0;
        for (int ch = 0; ch < nch; ++ch) {
            const int q0 = ch * kC, ct = min(kC, nk - q0), slot = ch % kR;
            bool ok = true;
            if (lane < ct) {
                const uint32_t a = offs[q0 + lane], e = offs[q0 + lane + 1];
                ok = e >= a && (e - a) <= (uint32_t)(kTM * kTK) && (a & 7u) == 0 && (e & 7u) == 0 &&
                     (uint64_t)e * 2u <= p.values_bytes;
            }
            const bool all_ok = __all_sync(0xffffffffu, ok);
            int fail = 0;
            if (lane == 0) {
                const uint32_t vb = all_ok ? (offs[q0 + ct] - offs[q0]) * 2u : 0u;
                const uint32_t sz = (uint32_t)ct * kBm + vb;
                // room for sz bytes: the ring holds chunks [tail, ch) in order
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
                    us::bulk_g2s(ring + place, p.bitmap + (tile0 + q0) * (kBm / 8), (uint32_t)ct * kBm, &S.full[slot]);
                    if (vb) us::bulk_g2s(ring + place + ct * kBm, p.values + (uint64_t)offs[q0] * 2u, vb, &S.full[slot]);
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
        if (early) us::pdl_wait();
    } else {
        // ----------------------------------------------------------- consumers
        us::pdl_wait();                                    // the activations may come from the previous kernel
        if (warp == 0 && lane == 0) {
            us::mbar_arrive_expect_tx(&S.xfull, (uint32_t)nk * kTK * 2u);
            us::bulk_g2s(xs, reinterpret_cast<const uint16_t*>(p.X) + (int64_t)kt0 * kTK, (uint32_t)nk * kTK * 2u,
                         &S.xfull);
        }
        bool ok = us::mbar_wait(&S.xfull, 0u, p.status);
        if (!ok) S.abort = 1;
        uint8_t* wbase = smem + L.warps + (uint32_t)warp * kWarpBytes;
        uint8_t* strip = wbase;                            // 32 columns x 128 B
        ColEnt* table = reinterpret_cast<ColEnt*>(wbase + kStrip);
        uint16_t* xc = reinterpret_cast<uint16_t*>(wbase + kStrip + kTable);   // compacted activations
        const uint32_t strip_s = us::smem_addr(strip);
        const uint32_t below = (1u << lane) - 1u;
        const int g = lane >> 2, tig = lane & 3;
        // ldmatrix row addresses: lane L supplies row (L & 7) of matrix L >> 3:
        // matrices 0..3 = (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7,
        // k 8-15), (rows 8-15, k 8-15) of a 16 x 16 A block
        const int lm_col = (lane & 7) + ((lane >> 4) << 3);   // compacted column of the group
        const int lm_half = (lane >> 3) & 1;                  // second 8 rows

        for (int q = warp; q < nk && ok; q += kNW) {
            const int ch = q / kC, slot = ch % kR;
            if (!us::mbar_wait(&S.full[slot], (uint32_t)(ch / kR) & 1u, p.status)) {
                S.abort = 1;
                ok = false;
                break;
            }
            const int ct = min(kC, nk - ch * kC);
            const uint8_t* base = ring + S.pos[slot];
            const uint64_t* bm = reinterpret_cast<const uint64_t*>(base + (q - ch * kC) * kBm);
            const uint32_t run_s = us::smem_addr(base + ct * kBm + (offs[q] - offs[ch * kC]) * 2u);
            const uint64_t wl = bm[lane], wh = bm[lane + 32];
            const uint32_t cl = (uint32_t)__popcll(wl), chh = (uint32_t)__popcll(wh);
            const uint32_t packed = cl | (chh << 16);
            uint32_t incl = packed;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += o;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t ex = incl - packed;
            const uint32_t totL = tot & 0xFFFFu;
            const bool good = S.bad[slot] == 0 && totL + (tot >> 16) <= offs[q + 1] - offs[q];
            if (!good && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
            const uint16_t xl = xs[q * kTK + lane], xh = xs[q * kTK + 32 + lane];
            const bool al = good && cl > 0 && fabsf(us::half_bits_to_float(xl)) > p.tau;
            const bool ah = good && chh > 0 && fabsf(us::half_bits_to_float(xh)) > p.tau;
            const uint32_t ml = __ballot_sync(0xffffffffu, al), mh = __ballot_sync(0xffffffffu, ah);
            const int a = __popc(ml) + __popc(mh);
            if (al)
                table[__popc(ml & below)] = ColEnt{(uint32_t)wl, (uint32_t)(wl >> 32), ex & 0xFFFFu,
                                                   (uint32_t)xl | ((uint32_t)__popc((uint32_t)wl) << 16)};
            if (ah)
                table[__popc(ml) + __popc(mh & below)] =
                    ColEnt{(uint32_t)wh, (uint32_t)(wh >> 32), totL + (ex >> 16),
                           (uint32_t)xh | ((uint32_t)__popc((uint32_t)wh) << 16)};
            __syncwarp();
            if (a == 0 && lane == 0) us::mbar_arrive(&S.empty[slot]);
            for (int g0 = 0; g0 < a; g0 += kGroup) {
                const int ag = min(kGroup, a - g0);
                // zero the strip and stage the group's activations (0 past its end)
#pragma unroll
                for (int i = lane; i < kGroup * 8; i += 32)
                    reinterpret_cast<uint4*>(strip)[i] = make_uint4(0u, 0u, 0u, 0u);
                if (lane < kGroup) xc[lane] = lane < ag ? (uint16_t)table[g0 + lane].x : (uint16_t)0;
                __syncwarp();
                // Each lane copies a share of one column's nonzeros: set bit i of
                // the column word is row i, its value the next one of the run;
                // 16-byte chunk k of column c sits at chunk k ^ (c & 7).
                if (ag <= 8) {
                    // four lanes per column: half-word h (rows 32 h ..), walked up
                    // from its first set bit (d = 0) or down from its last (d = 1),
                    // each for half of the half-word's set bits
                    const int c = lane & 7, h = (lane >> 3) & 1, d = lane >> 4;
                    if (c < ag) {
                        const ColEnt e = table[g0 + c];
                        const uint32_t w = h ? e.hi : e.lo;
                        const uint32_t n = (uint32_t)__popc(w);
                        const uint32_t first = e.base + (h ? (e.x >> 16) : 0u);
                        scatter_half(w, d ? n / 2u : (n + 1u) / 2u, d, run_s + 2u * (d ? first + n - 1u : first),
                                     (strip_s + (uint32_t)c * 128u) | (((uint32_t)h << 6) ^ ((uint32_t)(c & 7) << 4)));
                    }
                } else {
                    // two lanes per column: rows 0-31 (lanes 0-15), 32-63 (16-31),
                    // each walked down from its last set bit
                    const int c = lane & (kGroup - 1), h = lane >> 4;
                    if (c < ag) {
                        const ColEnt e = table[g0 + c];
                        const uint32_t w = h ? e.hi : e.lo;
                        const uint32_t n = (uint32_t)__popc(w);
                        scatter_half(w, n, 1, run_s + 2u * (e.base + (h ? (e.x >> 16) : 0u) + n - 1u),
                                     (strip_s + (uint32_t)c * 128u) | (((uint32_t)h << 6) ^ ((uint32_t)(c & 7) << 4)));
                    }
                }
                __syncwarp();
                // the tile's last columns are copied: its ring slot is free
                if (g0 + kGroup >= a && lane == 0) us::mbar_arrive(&S.empty[slot]);
                // B: the group's compacted activations (one K16 block) as token 0
                uint32_t b0 = 0u, b1 = 0u;
                if (g == 0) {
                    b0 = *reinterpret_cast<const uint32_t*>(xc + 2 * tig);
                    b1 = *reinterpret_cast<const uint32_t*>(xc + 8 + 2 * tig);
                }
#pragma unroll
                for (int mb = 0; mb < 4; ++mb) {
                    const uint32_t chunk = (uint32_t)(2 * mb + lm_half) ^ (uint32_t)(lm_col & 7);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_trans(strip_s + (uint32_t)lm_col * 128u + (chunk << 4), a0, a1, a2, a3);
                    us::mma_m16n8k16_f16(acc[mb], a0, a1, a2, a3, b0, b1);
                }
                __syncwarp();                              // the strip is refilled next
            }
        }
    }
    __syncthreads();
    if (S.abort && warp == kNW && lane == 0) {
        // a wait gave up: let the copies still in flight land (bounded); this
        // call's outputs are not valid (US_ERR_TIMEOUT is recorded)
        for (int ch = tail; ch < issued; ++ch) us::mbar_wait(&S.full[ch % kR], (uint32_t)(ch / kR) & 1u, nullptr);
        us::mbar_wait(&S.xfull, 0u, nullptr);
    }
    // ---- token 0 of the accumulators: thread (g, 0) holds rows 16 mb + g (c0)
    // and 16 mb + g + 8 (c2)
    if (warp < kNW && (lane & 3) == 0) {
        const int gg = lane >> 2;
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
            red[warp * kTM + 16 * mb + gg] = acc[mb][0];
            red[warp * kTM + 16 * mb + gg + 8] = acc[mb][2];
        }
    }
    __syncthreads();
    float* outv = red + kNW * kTM;
    for (int i = threadIdx.x; i < kTM; i += kThreads) {
        float s = 0.f;
        for (int w = 0; w < kNW; ++w) s += red[w * kTM + i];
        outv[i] = s;
    }
    __syncthreads();
    if (p.split > 1) {
        us::cluster_sync();
        const int rank = (int)us::cluster_ctarank();
        const int i0 = rank * kTM / p.split, i1 = (rank + 1) * kTM / p.split;
        for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
            float s = 0.f;
            for (int r = 0; r < p.split; ++r) s += us::ld_cluster_f32(us::cluster_map(outv + i, (uint32_t)r));
            p.Y[(int64_t)band * kTM + i] = us::float_to_half_bits(s);
        }
        us::cluster_sync();
    } else {
        for (int i = threadIdx.x; i < kTM; i += kThreads) p.Y[(int64_t)band * kTM + i] = us::float_to_half_bits(outv[i]);
    }
}

constexpr size_t kSmemPerCta = 74 * 1024;      // three CTAs of this size share one SM

}  // namespace

namespace us {

// K slices for the streamed kernel: the fewest (a cluster of at most 8) that
// give at least two CTAs per SM, so the three that fit on each SM keep its
// share of the stream even; each slice stages at most kMaxNk K tiles of
// activations.  0: not supported.
int spmspv_stream_split(int TM, int TK, int nTM, int nTK) {
    if (TM != kTM || TK != kTK) return 0;
    int s = 1;
    while (s < 8 && (nTK + s - 1) / s > kMaxNk) s *= 2;
    if ((nTK + s - 1) / s > kMaxNk) return 0;
    while (s < 8 && (int64_t)nTM * s < 2 * num_sms() && nTK / (2 * s) >= 2) s *= 2;
    if (s > nTK) s = nTK;
    return s;
}

us_status launch_spmspv_stream(UsKParams p, cudaStream_t st) {
    const int nk_max = (p.nTK + p.split - 1) / p.split;
    if (nk_max > kMaxNk) return US_ERR_UNSUPPORTED;
    const SvLayout L = sv_layout(nk_max);
    size_t ring = kSmemPerCta > L.ring + (size_t)kMinRing ? kSmemPerCta - L.ring : (size_t)kMinRing;
    ring &= ~(size_t)15;
    const size_t smem = L.ring + ring;
    p.sk_ring = (int)ring;
    auto kern = spmspv_stream_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nTM * p.split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace us
