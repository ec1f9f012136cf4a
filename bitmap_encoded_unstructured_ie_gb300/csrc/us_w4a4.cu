// us_w4a4.cu -- W4A4 bitmap SpMM on CUDA cores for decode-sized token counts.
//
// Y = W . X with W int4 in 64 x 64 bitmap tiles, row-major scan (IE-BME of
// "UnionSparse: An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM
// Inference on Edge", section V-A, one area), X int4 per token, int32
// accumulation, dequantised fp16 epilogue (same page, Fig. 2).
//
// GB300 design (the page's LSPD/DW-PC kernel targets Ampere mma.sync; here the
// decode feeds dp4a directly and the kernel is built around latency):
//  * the tiles of one K slice of a band are consecutive in the bitmap and in
//    the value array, so one producer warp moves up to eight tiles with two
//    1-D bulk copies (TMA): the bitmap words and the concatenated 16-byte
//    padded nibble runs.  Chunks of eight tiles alternate between two
//    shared-memory buffers with "full"/"empty" mbarriers (the
//    producer/consumer split of UnionSparse's DW-PC pipeline, section VI-A);
//  * meanwhile the consumer warps build the byte-selector table and expand
//    this CTA's activations to int8 in shared memory;
//  * each consumer warp owns whole tiles; lane l decodes rows l and l+32 (one
//    64-bit bitmap word each).  The row bases - popcounts of the earlier rows,
//    the word-level part of UnionSparse's idx_base (section VI-B) - come from
//    one warp scan of packed popcounts;
//  * a row word is walked one byte (8 positions) at a time.  A funnel-shift
//    window over the row's nibble stream, masked to popc(byte) nibbles, is
//    split into even and odd ranks placed in the high nibble of each byte
//    (each byte then holds 16*w as a signed int8); one PRMT per 4 positions,
//    with a selector looked up by the byte value, moves rank r to its position
//    and fills clear positions from the masked, zero rank-7 byte;
//  * dp4a against the int8 activations; accumulators hold 16 * sum and are
//    shifted back exactly at the end;
//  * split-K without global memory: the K slices of a band are one thread-block
//    cluster; after a cluster barrier each CTA sums its share of the outputs
//    over every slice straight from the other CTAs' shared memory (integer
//    adds: exact) and writes Yacc and the fp16 output;
//  * launched with programmatic stream serialisation: the barrier and table
//    set-up overlap the previous kernel's tail; activations and outputs are
//    touched only after griddepcontrol.wait, and so are the weights unless the
//    caller marked them static (then their bulk copies start right away).
#include "us_common.cuh"
#include "us_internal.h"

#ifndef US_W4A4_CONSUMERS
#define US_W4A4_CONSUMERS 4          // consumer warps per CTA
#endif
#ifndef US_W4A4_CTAS_PER_SM
#define US_W4A4_CTAS_PER_SM 2        // split-K target: this many CTAs per SM
#endif

namespace {

constexpr int kTM = 64, kTK = 64;
constexpr int kChunk = 8;                               // tiles per bulk-copy chunk
constexpr int kBmBytes = kTM * kTK / 8;                 // 512 per tile
constexpr int kValCap = kTM * kTK / 2;                  // 2048 per tile
constexpr int kBufBytes = kChunk * (kBmBytes + kValCap);   // 20480 per chunk buffer
constexpr int kLutRep = 16;                             // LUT replicas (bank spreading)
constexpr int kHeader = 256;

struct Smem {
    uint64_t full[2];
    uint64_t empty[2];
    uint32_t bad[2];              // chunk in buffer b failed its offset checks
    uint32_t abort;
};
static_assert(sizeof(Smem) <= kHeader, "header");

constexpr int threads_for(int NC) { return (NC + 1) * 32; }

// N tokens per CTA (blockIdx.y selects the token block), NC consumer warps.
template <int N, int NC>
__global__ void __launch_bounds__(threads_for(NC))
w4a4_small_n_kernel(const UsKParams p) {
    constexpr int kThreads = threads_for(NC);
    constexpr int kConsumerThreads = NC * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    Smem& S = *reinterpret_cast<Smem*>(smem);
    uint8_t* bufs = smem + kHeader;
    const int band = blockIdx.x / p.split;               // the split slices of a band form one cluster
    const int slice = blockIdx.x % p.split;
    const int kt0 = (int)((int64_t)slice * p.nTK / p.split);
    const int kt1 = (int)((int64_t)(slice + 1) * p.nTK / p.split);
    const int nk = kt1 - kt0;
    const int nchunks = (nk + kChunk - 1) / kChunk;
    const int nbuf = nchunks > 1 ? 2 : 1;
    uint32_t* lut = reinterpret_cast<uint32_t*>(bufs + nbuf * kBufBytes + 16);   // 256 x kLutRep
    uint32_t* offs = lut + 256 * kLutRep;                                         // nk + 1
    const int krange = nk * kTK;
    int8_t* xs = reinterpret_cast<int8_t*>(offs + ((nk + 1 + 3) & ~3));          // N x krange int8
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tile0 = (int64_t)band * p.nTK + kt0;
    const int tok0 = blockIdx.y * N;                     // first token of this CTA
    const int ntok = min(N, p.N - tok0);                 // tokens present (ragged last block)
    const bool early = (p.flags & US_BITMAP_STATIC) != 0; // weights may be fetched before the wait

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            us::mbar_init(&S.full[b], 1);
            us::mbar_init(&S.empty[b], NC);
        }
        S.abort = 0;
        us::fence_mbar_init();
    }
    __syncthreads();
    // every thread of every CTA: the next launch may begin its own prologue now
    // (it reads nothing of ours before its griddepcontrol.wait)
    us::pdl_launch_dependents();

    int issued = 0;                                      // chunks issued (producer lane 0)
    if (warp == NC) {
        // ---------------------------------------------------------- producer
        if (!early) us::pdl_wait();
        for (int q = lane; q <= nk; q += 32) offs[q] = p.tile_off[tile0 + q];
        __syncwarp();
        for (int c = 0; c < nchunks; ++c) {
            const int b = c & 1;
            const int q0 = c * kChunk, ct = min(kChunk, nk - q0);
            bool ok = true;
            if (lane < ct) {
                const uint32_t o0 = offs[q0 + lane], o1 = offs[q0 + lane + 1];
                ok = o1 >= o0 && (o1 - o0) <= (uint32_t)(kTM * kTK) && (o0 & 31u) == 0 && (o1 & 31u) == 0 &&
                     (uint64_t)o1 * 4u <= p.values_bytes * 8ull;
            }
            const bool all_ok = __all_sync(0xffffffffu, ok);
            // the consumers start only after the previous launch has finished: wait
            // for that too before a bounded wait on them
            if (c == 2 && early) us::pdl_wait();
            if (lane == 0) {
                if (c >= 2 && !us::mbar_wait(&S.empty[b], ((c >> 1) - 1) & 1, p.status)) {
                    S.abort = 1;
                } else {
                    if (!all_ok) us::set_status(p.status, US_ERR_CORRUPT);
                    const uint32_t vbytes = all_ok ? (offs[q0 + ct] - offs[q0]) / 2u : 0u;
                    S.bad[b] = all_ok ? 0u : 1u;
                    uint8_t* dst = bufs + b * kBufBytes;
                    us::mbar_arrive_expect_tx(&S.full[b], (uint32_t)ct * kBmBytes + vbytes);
                    us::bulk_g2s(dst, p.bitmap + (tile0 + q0) * (kTM * kTK / 64), (uint32_t)ct * kBmBytes,
                                 &S.full[b]);
                    if (vbytes) us::bulk_g2s(dst + kChunk * kBmBytes, p.values + offs[q0] / 2u, vbytes, &S.full[b]);
                    issued = c + 1;
                }
            }
            if (__shfl_sync(0xffffffffu, S.abort, 0)) break;
        }
    }

    int acc[2][N];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int n = 0; n < N; ++n) acc[h][n] = 0;

    if (warp < NC) {
        // ---------------------------------------------------------- consumers
        // selector table, kLutRep copies (bank spreading)
        for (int e = threadIdx.x; e < 256; e += kConsumerThreads) {
            const uint32_t sel = us::make_sel((uint32_t)e);
#pragma unroll
            for (int r = 0; r < kLutRep; ++r) lut[e * kLutRep + r] = sel;
        }
        us::pdl_wait();
        // activations of this CTA's K range: 8 nibbles -> 8 sign-extended bytes
        {
            const uint8_t* xg = reinterpret_cast<const uint8_t*>(p.X);
            const int words_per_tok = krange / 8;
            for (int i = threadIdx.x; i < N * words_per_tok; i += kConsumerThreads) {
                const int n = i / words_per_tok, w = i - n * words_per_tok;
                const uint32_t v = n < ntok ? __ldg(reinterpret_cast<const uint32_t*>(
                                                  xg + ((int64_t)(tok0 + n) * p.K + (int64_t)kt0 * kTK) / 2 + 4 * w))
                                            : 0u;                        // absent tokens: zero activations
                const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;
                const uint32_t e0 = __vsub4(__byte_perm(lo, hi, 0x5140) ^ 0x08080808u, 0x08080808u);
                const uint32_t e1 = __vsub4(__byte_perm(lo, hi, 0x7362) ^ 0x08080808u, 0x08080808u);
                *reinterpret_cast<uint2*>(xs + (int64_t)n * krange + 8 * w) = make_uint2(e0, e1);
            }
        }
        us::named_bar_sync(1, kConsumerThreads);

        const uint32_t lut_lane = (uint32_t)(lane % kLutRep);
        for (int c = 0; c < nchunks; ++c) {
            const int b = c & 1;
            const int q0 = c * kChunk, ct = min(kChunk, nk - q0);
            if (!us::mbar_wait(&S.full[b], (c >> 1) & 1, p.status)) {
                S.abort = 1;
                break;
            }
            const uint8_t* buf = bufs + b * kBufBytes;
            const bool chunk_ok = S.bad[b] == 0;
            for (int qq = warp; qq < ct; qq += NC) {
                const int q = q0 + qq;
                const uint64_t* bm = reinterpret_cast<const uint64_t*>(buf + qq * kBmBytes);
                const uint32_t* vw = reinterpret_cast<const uint32_t*>(buf + kChunk * kBmBytes +
                                                                        (offs[q] - offs[q0]) / 2u);
                const uint64_t wA = bm[lane], wB = bm[lane + 32];
                const uint32_t cA = __popcll(wA), cB = __popcll(wB);
                const uint32_t packed = cA | (cB << 16);
                uint32_t incl = packed;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += o;
                }
                const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
                const uint32_t ex = incl - packed;
                const uint32_t totA = tot & 0xFFFFu;
                const uint32_t P = totA + (tot >> 16);
                const bool good = chunk_ok && P <= offs[q + 1] - offs[q];
                if (!good && lane == 0) us::set_status(p.status, US_ERR_CORRUPT);
                if (!good) continue;
                const int8_t* xt = xs + (q * kTK);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint64_t w = h ? wB : wA;
                    const uint32_t o = h ? totA + (ex >> 16) : (ex & 0xFFFFu);
                    const uint32_t lo = (uint32_t)w, hi = (uint32_t)(w >> 32);
                    const uint32_t plo = (uint32_t)__popc(lo);
                    // eight independent byte-steps: each finds its own place in the
                    // run (row base + popcount of the lower bits), so all are in flight
#pragma unroll
                    for (int bt = 0; bt < 8; ++bt) {
                        const uint32_t bb = ((bt < 4 ? lo : hi) >> (8 * (bt & 3))) & 0xFFu;
                        const uint32_t below =
                            bt == 0 ? 0u
                                    : (bt < 4 ? (uint32_t)__popc(lo & ((1u << (8 * bt)) - 1u))
                                              : plo + (bt == 4 ? 0u : (uint32_t)__popc(hi & ((1u << (8 * (bt - 4))) - 1u))));
                        const uint32_t ob = o + below;
                        const uint32_t sel = lut[bb * kLutRep + lut_lane];
                        const uint32_t c4 = (uint32_t)__popc(bb) << 2;
                        const uint32_t wi = ob >> 3;
                        const uint32_t nm = __funnelshift_r(vw[wi], vw[wi + 1], ob << 2) &
                                            ~us::shl_clamp(0xFFFFFFFFu, c4);           // first c nibbles
                        const uint32_t odd = nm & 0xF0F0F0F0u;                   // 16 * w of ranks 1,3,5,7
                        const uint32_t even = (nm << 4) & 0xF0F0F0F0u;           // 16 * w of ranks 0,2,4,6
                        const int d0 = (int)__byte_perm(even, odd, sel);
                        const int d1 = (int)__byte_perm(even, odd, sel >> 16);
#pragma unroll
                        for (int n = 0; n < N; ++n) {
                            const uint2 xv = *reinterpret_cast<const uint2*>(xt + (int64_t)n * krange + 8 * bt);
                            acc[h][n] = __dp4a(d0, (int)xv.x, acc[h][n]);
                            acc[h][n] = __dp4a(d1, (int)xv.y, acc[h][n]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) us::mbar_arrive(&S.empty[b]);
        }
    }
    __syncthreads();
    if (S.abort && warp == NC && lane == 0) {
        // a wait gave up: let the copies still in flight land (bounded); the
        // outputs of this call are not valid (US_ERR_TIMEOUT is recorded)
        for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
            us::mbar_wait(&S.full[c & 1], (c >> 1) & 1, nullptr);
    }
    if (warp == NC && early) us::pdl_wait();              // before the first global write

    // ---- reduce the consumer warps in fixed order
    int* red = reinterpret_cast<int*>(bufs);             // NC x N x 64 (the chunk buffers are idle now)
    if (warp < NC) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            red[(warp * N + n) * kTM + lane] = acc[0][n];
            red[(warp * N + n) * kTM + lane + 32] = acc[1][n];
        }
    }
    __syncthreads();
    int* outv = red + NC * N * kTM;                      // N x 64 partial of this K slice
    for (int i = threadIdx.x; i < N * kTM; i += kThreads) {
        int v = 0;
#pragma unroll
        for (int w = 0; w < NC; ++w) v += red[w * N * kTM + i];
        outv[i] = v >> 4;                                 // exact: every term is 16 * w * x
    }
    __syncthreads();

    // ---- split-K: the slices of a band are one cluster; rank r sums every
    // slice's partial for its share of the outputs straight from the other
    // CTAs' shared memory (integer adds: exact), then writes Yacc and Y.
    const int m0 = band * kTM;
    auto store = [&](int i, int a) {
        const int nl = i / kTM, r = i - nl * kTM;
        if (nl >= ntok) return;
        const int n = tok0 + nl, m = m0 + r;
        const int64_t o = (int64_t)n * p.M + m;
        p.Yacc[o] = a;
        if (p.Y) {
            const float t = __fmul_rn(__int2float_rn(a), us::half_bits_to_float(p.s_w[m]));
            p.Y[o] = us::float_to_half_bits(__fmul_rn(t, us::half_bits_to_float(p.s_x[n])));
        }
    };
    if (p.split > 1) {
        us::cluster_sync();
        const int rank = (int)us::cluster_ctarank();
        // rank r reduces elements [r*total/split, (r+1)*total/split): any split, no remainder lost
        const int i0 = rank * (N * kTM) / p.split, i1 = (rank + 1) * (N * kTM) / p.split;
        for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
            int a = 0;
            for (int r = 0; r < p.split; ++r) a += us::ld_cluster_s32(us::cluster_map(outv + i, (uint32_t)r));
            store(i, a);
        }
        us::cluster_sync();                               // no CTA leaves while others read its partial
    } else {
        for (int i = threadIdx.x; i < N * kTM; i += kThreads) store(i, outv[i]);
    }
}

size_t smem_bytes(int N, int nk) {
    const int nbuf = nk > kChunk ? 2 : 1;
    const size_t base = kHeader + (size_t)nbuf * kBufBytes + 16 + 256 * kLutRep * 4;
    const size_t offs = (size_t)((nk + 1 + 3) & ~3) * 4;
    const size_t xs = (size_t)N * nk * kTK;
    return base + offs + xs;
}

template <int N, int NC>
us_status launch_n(const UsKParams& p, cudaStream_t st) {
    static_assert((NC + 1) * 8 * kTM * 4 <= kBufBytes, "reduction buffers must fit a chunk buffer");
    const int nk = (p.nTK + p.split - 1) / p.split;
    const size_t smem = smem_bytes(N, nk);
    if (smem > 200 * 1024) return US_ERR_UNSUPPORTED;
    auto kern = w4a4_small_n_kernel<N, NC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return US_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nTM * p.split), (unsigned)((p.N + N - 1) / N));
    cfg.blockDim = dim3(threads_for(NC));
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

constexpr int kNC = US_W4A4_CONSUMERS;

}  // namespace

namespace us {

constexpr int kMaxN = 32;      // token counts above this use the tensor-core / general path

bool w4a4_fast_supported(int TM, int TK, int N) { return TM == kTM && TK == kTK && N >= 1 && N <= kMaxN; }

int w4a4_fast_tok_block(int N) { return N <= 8 ? N : 8; }

size_t w4a4_fast_ws(int, int, int, int) { return 0; }     // split-K reduces inside the cluster

int w4a4_fast_max_split() { return 8; }                      // portable cluster size

int w4a4_fast_target_ctas() { return US_W4A4_CTAS_PER_SM * num_sms(); }

us_status launch_w4a4_fast(const UsKParams& p, cudaStream_t st) {
    switch (w4a4_fast_tok_block(p.N)) {
        case 1: return launch_n<1, kNC>(p, st);
        case 2: return launch_n<2, kNC>(p, st);
        case 3: return launch_n<3, kNC>(p, st);
        case 4: return launch_n<4, kNC>(p, st);
        case 5: return launch_n<5, kNC>(p, st);
        case 6: return launch_n<6, kNC>(p, st);
        case 7: return launch_n<7, kNC>(p, st);
        case 8: return launch_n<8, kNC>(p, st);
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
