// us_f16_dec.cu -- fp16 SpMM for decode-sized token counts (1-63 tokens) on
// 64 x 64 bitmap tiles with the row-major scan.
//
// Y = W . X with W fp16 in bitmap tiles (IE-BME of "UnionSparse: An
// Index-Efficient Sparsity Framework for Low-Bit Sparse LLM Inference on
// Edge", section V-A, one area; bit p = i*64 + j of a tile marks W[i][j] != 0
// and the nonzeros follow in p order from the tile's offset).  fp32
// accumulation, one fp16 rounding at the end.
//
// Per CTA: one 64-row band x one K slice x one block of 8, 16 or 32 tokens;
// eight warps in two groups of four.  A group takes every other tile of the
// slice and its four warps decode the same tile together, one 16-row strip
// each.  Each group runs a three-stage ring (two stages when three CTAs share
// an SM, for grids of more than one wave at two): one lane issues, per tile, a bulk
// copy of the 512-byte bitmap, a bulk copy of the value run (16-byte padded,
// its length from the offset array) and a 2-D TMA load of the 64-column
// activation tile for the token block (128-byte swizzle), all completing on
// the stage's full barrier; the four warps release the stage on its empty
// barrier.  This is the prefetch/compute overlap of UnionSparse's DW-PC
// pipeline (section VI-A) with the bulk-copy engine doing the prefetch.
//
// Decode (UnionSparse section VI-B, rank addressing): every warp scans the
// 64 row popcounts for the row prefixes; then, two rows per step, lane l
// takes four adjacent columns 4 (l % 16) .. + 3 of row 2 j + l / 16.  The
// rank of the first is the row prefix plus the popcount of the row word's
// lower bits, the next ones follow by the nibble's own bits, and the four
// values leave as one 8-byte store into a dense 16 x 64 strip whose 16-byte
// chunks are swizzled by row.  The strip feeds ldmatrix + mma.sync m16n8k16
// (fp16 x fp16 -> fp32) against the activation fragments, loaded once per
// tile.  A warp's accumulators cover its 16 rows of the band for all the
// block's tokens, so nothing is reduced per tile: the two groups' sums are
// added once at the end, and split-K partials follow the generic kernel's
// deterministic protocol (the last CTA of a band adds the slices in slice
// order and clears them).
//
// Launches overlap (programmatic dependent launch): a CTA starts while the
// previous kernel drains; with US_BITMAP_STATIC weights its issuing lanes
// request the first stages' bitmaps and value runs before the dependency
// wait and the activation tiles after it; nothing else global is read or
// written before the wait.
//
// Every wait is bounded (US_ERR_TIMEOUT); offsets that are not a valid run
// and runs shorter than their bitmap's popcount record US_ERR_CORRUPT and
// the tile is skipped, so no access leaves its buffer.
#include <cudaTypedefs.h>

#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kGroups = 2;                      // warp groups, each on its own tiles
constexpr int kGroupWarps = 4;                  // one 16-row strip of the tile each
constexpr int kWarps = kGroups * kGroupWarps;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;                      // per group, at most (two CTAs an SM)
constexpr uint32_t kBmBytes = 512;              // 64 words of a 64 x 64 tile
constexpr uint32_t kRunCap = 64 * 64 * 2;       // a full tile of fp16 values
constexpr uint32_t kStripBytes = 16 * 128;      // 16 rows x 64 fp16
constexpr uint32_t kHeader = 2048;

template <int NB>
struct DecShape {
    static constexpr int kTB = 8 * NB;                          // tokens per CTA
    static constexpr uint32_t kXBytes = kTB * 128;              // activation tile (1024-aligned)
    static constexpr uint32_t kStage = (kXBytes + kBmBytes + kRunCap + 1023u) & ~1023u;
};

struct DecHeader {
    uint64_t full[kGroups][kStages];   // the stage's copies have landed
    uint64_t empty[kGroups][kStages];  // the group's four warps are done reading it
    uint32_t len[kGroups][kStages];    // run length of the staged tile (elements)
    uint32_t pre[kWarps][16];          // prefixes of the warp's 16 rows in its current tile
    int flag;
};
static_assert(sizeof(DecHeader) <= kHeader, "header");

US_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// 2-D TMA tile load (x = K element, y = token) completing on `bar`
US_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(us::smem_addr(bar))
        : "memory");
}

// three CTAs an SM (grids of more than one wave at two) keep two stages a group
__host__ __device__ constexpr int stages_for(int minb) { return minb >= 3 ? 2 : kStages; }

size_t dec_smem(int nk, int NB, int stages = kStages) {
    const uint32_t stage = ((uint32_t)(8 * NB) * 128u + kBmBytes + kRunCap + 1023u) & ~1023u;
    const size_t offs = (((size_t)nk + 1) * 4 + 1023) & ~(size_t)1023;
    return 1024 + kHeader + offs + (size_t)kGroups * stages * stage + (size_t)kWarps * kStripBytes;
}

template <int NB, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
spmm_f16_dec_kernel(const UsKParams p, const __grid_constant__ CUtensorMap xmap) {
    using S = DecShape<NB>;
    constexpr int kSt = stages_for(MINB);              // stages a group
    constexpr int TB = S::kTB;
    extern __shared__ uint8_t smem_raw[];
    // the swizzled TMA destinations want 1024-byte alignment
    uint8_t* smem = smem_raw + ((1024u - (us::smem_addr(smem_raw) & 1023u)) & 1023u);
    DecHeader& h = *reinterpret_cast<DecHeader*>(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp / kGroupWarps, sw = warp % kGroupWarps;    // group, strip (rows 16 sw ..)
    const int band = blockIdx.x % p.nTM, slice = blockIdx.x / p.nTM, tb = blockIdx.y;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int64_t tile0 = (int64_t)band * p.nTK + kt0;

    uint32_t* offs = reinterpret_cast<uint32_t*>(smem + kHeader);
    const uint32_t offs_bytes = ((uint32_t)(nk + 1) * 4u + 1023u) & ~1023u;
    uint8_t* stages = smem + kHeader + offs_bytes;
    uint8_t* strip_g = stages + kGroups * kSt * S::kStage + warp * kStripBytes;
    const uint32_t strip = us::smem_addr(strip_g);

    const bool early = (p.flags & US_BITMAP_STATIC) != 0;   // weights may be fetched before the wait
    if (!early) us::pdl_wait();
    for (int q = threadIdx.x; q <= nk; q += kThreads) offs[q] = p.tile_off[tile0 + q];
    if (threadIdx.x < kGroups * kSt) {
        us::mbar_init(&h.full[threadIdx.x / kSt][threadIdx.x % kSt], 1);
        us::mbar_init(&h.empty[threadIdx.x / kSt][threadIdx.x % kSt], kGroupWarps);
    }
    us::fence_mbar_init();
    __syncthreads();
    us::pdl_launch_dependents();

    // the group's tiles: q = grp + kGroups * r, r = 0 .. nr - 1
    const int nr = nk > grp ? (nk - grp + kGroups - 1) / kGroups : 0;
    uint8_t* gstages = stages + grp * kSt * S::kStage;
    const bool issuer = sw == 0 && lane == 0;

    // a stage's three copies complete on its full barrier: the weights
    // (bitmap, value run; the barrier expects all three) and the activations
    auto issue_w = [&](int r) {          // the group's issuing lane only
        const int st = r % kSt;
        const int q = grp + kGroups * r;
        uint8_t* sp = gstages + st * S::kStage;
        const uint32_t o0 = offs[q], o1 = offs[q + 1];
        const bool ok = o1 >= o0 && o1 - o0 <= kRunCap / 2u && (o0 & 7u) == 0 && (o1 & 7u) == 0 &&
                        (uint64_t)o1 * 2u <= p.values_bytes;
        if (!ok) us::set_status(p.status, US_ERR_CORRUPT);
        const uint32_t len = ok ? o1 - o0 : 0u;
        h.len[grp][st] = len;
        us::mbar_arrive_expect_tx(&h.full[grp][st], S::kXBytes + kBmBytes + len * 2u);
        us::bulk_g2s(sp + S::kXBytes, p.bitmap + (tile0 + q) * 64, kBmBytes, &h.full[grp][st]);
        if (len) us::bulk_g2s(sp + S::kXBytes + kBmBytes, p.values + (uint64_t)o0 * 2u, len * 2u, &h.full[grp][st]);
    };
    auto issue_x = [&](int r) {
        const int st = r % kSt;
        const int q = grp + kGroups * r;
        tma_load_2d(us::smem_addr(gstages + st * S::kStage), &xmap, (kt0 + q) * 64, tb * TB, &h.full[grp][st]);
    };
    if (issuer)
        for (int r = 0; r < nr && r < kSt; ++r) issue_w(r);
    // everything below reads the activations or writes global memory
    if (early) us::pdl_wait();
    if (issuer)
        for (int r = 0; r < nr && r < kSt; ++r) issue_x(r);

    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;

    // decode lanes: row 2 j + rr of a row pair, columns 4 c4 .. 4 c4 + 3
    const int rr = lane >> 4, c4 = lane & 15;
    const uint64_t below = (1ull << (4 * c4)) - 1ull;
    bool failed = false;
    for (int r = 0; r < nr; ++r) {
        const int st = r % kSt;
        const uint32_t ph = (uint32_t)(r / kSt) & 1u;
        uint8_t* sp = gstages + st * S::kStage;
        if (!__all_sync(0xffffffffu, us::mbar_wait(&h.full[grp][st], ph, p.status))) {
            // give each copy that may still be in flight one more bounded wait, then stop
            for (int r2 = r + 1; r2 < nr && r2 < r + kSt; ++r2)
                us::mbar_wait(&h.full[grp][r2 % kSt], (uint32_t)(r2 / kSt) & 1u, nullptr);
            failed = true;
            break;
        }
        const uint64_t* words = reinterpret_cast<const uint64_t*>(sp + S::kXBytes);
        const uint16_t* run = reinterpret_cast<const uint16_t*>(sp + S::kXBytes + kBmBytes);
        const uint32_t len = h.len[grp][st];

        // 1. row prefixes: a warp scan of the 64 row popcounts (two rows a
        //    lane); this warp keeps those of its own 16 rows
        const uint64_t w0 = words[2 * lane], w1 = words[2 * lane + 1];
        const int c0 = __popcll(w0), c1 = __popcll(w1);
        const int incl = us::warp_incl_scan(c0 + c1);
        const uint32_t P = (uint32_t)__shfl_sync(0xffffffffu, incl, 31);
        const bool tile_ok = P <= len;
        if (!tile_ok && sw == 0 && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
        if ((lane >> 3) == sw) {
            h.pre[warp][2 * (lane & 7)] = (uint32_t)(incl - c0 - c1);
            h.pre[warp][2 * (lane & 7) + 1] = (uint32_t)(incl - c1);
        }

        // 2. activation fragments of the tile: matrix rows are tokens, each
        //    holding 8 consecutive columns (128-byte swizzle: chunk ^ token % 8)
        uint32_t b[NB][4][2];
        const uint32_t xs = us::smem_addr(sp);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t n = 8 * nb + (lane & 7);
                const uint32_t chunk = 4 * h2 + (lane >> 3);
                ldsm_x4(xs + n * 128 + ((chunk ^ (n & 7)) << 4), b[nb][2 * h2][0], b[nb][2 * h2][1],
                        b[nb][2 * h2 + 1][0], b[nb][2 * h2 + 1][1]);
            }
        __syncwarp();

        // 3. decode the warp's 16 rows into a dense strip (row i, 16-byte
        //    chunk c at c ^ (i % 8)), two rows per step, four rows' loads in
        //    flight before their stores
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint64_t w[4];
            uint32_t pr[4], v01[4], v23[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = 8 * hb + 2 * j + rr;
                w[j] = tile_ok ? words[16 * sw + i] : 0ull;
                pr[j] = h.pre[warp][i];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t k = pr[j] + (uint32_t)__popcll(w[j] & below);
                const uint32_t nib = (uint32_t)(w[j] >> (4 * c4)) & 15u;
                uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
                if (nib & 1u) a0 = run[k];
                k += nib & 1u;
                if (nib & 2u) a1 = run[k];
                k += (nib >> 1) & 1u;
                if (nib & 4u) a2 = run[k];
                k += (nib >> 2) & 1u;
                if (nib & 8u) a3 = run[k];
                v01[j] = a0 | (a1 << 16);
                v23[j] = a2 | (a3 << 16);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = 8 * hb + 2 * j + rr;
                uint2* d = reinterpret_cast<uint2*>(strip_g + i * 128 + ((((uint32_t)c4 >> 1) ^ (uint32_t)(i & 7)) << 4) +
                                                    ((c4 & 1) << 3));
                *d = make_uint2(v01[j], v23[j]);
            }
        }

        // 4. this warp is done with the stage; the issuing lane refills it
        //    once all four warps of the group are
        __syncwarp();
        if (lane == 0) us::mbar_arrive(&h.empty[grp][st]);
        if (issuer && r + kSt < nr) {
            if (us::mbar_wait(&h.empty[grp][st], ph, p.status)) {
                issue_w(r + kSt);
                issue_x(r + kSt);
            }
        }
        __syncwarp();                           // reconverge before the warp-wide ldmatrix / mma

        // 5. multiply the strip
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
            const uint32_t row = (lane & 7) + 8 * ((lane >> 3) & 1);
            const uint32_t chunk = 2 * kc + (lane >> 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(strip + row * 128 + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
                us::mma_m16n8k16_f16(acc[nb], a0, a1, a2, a3, b[nb][kc][0], b[nb][kc][1]);
        }
        __syncwarp();                           // the next tile's decode overwrites the strip
    }

    // ---- the two groups' sums, added in group order
    if (__syncthreads_or(failed)) return;
    float* red = reinterpret_cast<float*>(stages);     // [kGroups][TB][64]; every copy has landed
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float* rw = red + ((size_t)grp * TB + 8 * nb + 2 * t) * 64 + 16 * sw + g;
            rw[0] = acc[nb][0];
            rw[64] = acc[nb][1];
            rw[8] = acc[nb][2];
            rw[72] = acc[nb][3];
        }
    }
    __syncthreads();
    const int nTB = gridDim.y;
    const int m0 = band * 64;
    if (p.split > 1) {
        float* part = reinterpret_cast<float*>(p.ws);
        const int64_t base = (((int64_t)slice * nTB + tb) * p.nTM + band) * (int64_t)(TB * 64);
        for (int idx = threadIdx.x; idx < TB * 64; idx += kThreads) part[base + idx] = red[idx] + red[TB * 64 + idx];
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned old = atomicAdd(&p.counters[band * nTB + tb], 1u);
            h.flag = (old == (unsigned)p.split - 1u);
        }
        __syncthreads();
        if (!h.flag) return;
        __threadfence();
        for (int idx = threadIdx.x; idx < TB * 64; idx += kThreads) {
            float v = 0.f;
            for (int sl = 0; sl < p.split; ++sl) {
                float* src = part + (((int64_t)sl * nTB + tb) * p.nTM + band) * (int64_t)(TB * 64) + idx;
                v += __ldcg(src);
                __stcg(src, 0.f);               // leave the workspace zeroed for the next call
            }
            const int n = tb * TB + (idx >> 6);
            if (n < p.N) p.Y[(int64_t)n * p.M + m0 + (idx & 63)] = us::float_to_half_bits(v);
        }
        if (threadIdx.x == 0) p.counters[band * nTB + tb] = 0u;
    } else {
        for (int idx = threadIdx.x; idx < TB * 64; idx += kThreads) {
            const float v = red[idx] + red[TB * 64 + idx];
            const int n = tb * TB + (idx >> 6);
            if (n < p.N) p.Y[(int64_t)n * p.M + m0 + (idx & 63)] = us::float_to_half_bits(v);
        }
    }
}

template <int NB, int MINB>
us_status launch_nb(const UsKParams& p, cudaStream_t st) {
    auto enc = us::tensor_map_encoder();
    if (!enc) return US_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)p.K, (cuuint64_t)p.N};
    const cuuint64_t gstride[1] = {(cuuint64_t)p.K * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)(8 * NB)};
    const cuuint32_t estr[2] = {1, 1};
    // rows past the last token read as zeros
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(p.X), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return US_ERR_CUDA;
    const int nk = (p.nTK + p.split - 1) / p.split;
    const size_t smem = dec_smem(nk, NB, stages_for(MINB));
    if (smem > 227 * 1024) return US_ERR_UNSUPPORTED;
    auto kern = spmm_f16_dec_kernel<NB, MINB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nTM * p.split), (unsigned)((p.N + 8 * NB - 1) / (8 * NB)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, map) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace

namespace us {

bool f16_dec_supported(int TM, int TK, int order, int N) {
    return TM == 64 && TK == 64 && order == US_ORDER_ROW && N >= 1 && N < 64;
}

int f16_dec_tok_block(int N) { return N <= 8 ? 8 : (N <= 16 ? 16 : 32); }

bool f16_dec_fits(int nTK, int split, int N) {
    if (split < 1 || split > nTK) return false;
    return dec_smem((nTK + split - 1) / split, f16_dec_tok_block(N) / 8) <= 227 * 1024;
}

// K slices of about 16 tiles (eight per warp group: the shortest slices
// that still hide the copies' latency), more when the bands alone leave SMs
// idle
int f16_dec_split(int nTM, int nTK, int N) {
    const int tb = f16_dec_tok_block(N);
    const int ntb = (N + tb - 1) / tb;
    int s = 1;
    while (nTK / (2 * s) >= 16) s *= 2;
    while ((int64_t)nTM * s * ntb < num_sms() && nTK / (2 * s) >= 4) s *= 2;
    while (!f16_dec_fits(nTK, s, N) && s < nTK) s *= 2;
    return s > nTK ? nTK : s;
}

us_status launch_f16_dec(const UsKParams& p, cudaStream_t st) {
    // a grid of more than one wave at two CTAs an SM runs three an SM with two
    // stages a group (measured: 11008 x 4096, N = 1 / 16: 39.6 / 45.7 ->
    // 34.9 / 42.0 us); a smaller grid keeps the deeper ring (4096 x 4096, N =
    // 1: 17.1 us with it, 21.2 without)
    const int ntb = (p.N + p.tok_block - 1) / p.tok_block;
    const int nk = (p.nTK + p.split - 1) / p.split;
    const bool three = p.tok_block <= 16 && (int64_t)p.nTM * p.split * ntb > 2 * num_sms() &&
                       3 * (dec_smem(nk, p.tok_block / 8, stages_for(3)) + 1024) <= 228 * 1024;
    switch (p.tok_block) {
        case 8: return three ? launch_nb<1, 3>(p, st) : launch_nb<1, 2>(p, st);
        case 16: return three ? launch_nb<2, 3>(p, st) : launch_nb<2, 2>(p, st);
        case 32: return launch_nb<4, 2>(p, st);
    }
    return US_ERR_INVALID_ARG;
}

}  // namespace us
