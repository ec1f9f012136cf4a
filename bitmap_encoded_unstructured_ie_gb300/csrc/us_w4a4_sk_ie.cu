// us_w4a4_sk_ie.cu -- the balanced W4A4 kernel on IE-BME with areas ("UnionSparse:
// An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM Inference on
// Edge", section V-A with Q = RA x CA > 1 and the row reordering of section
// V-B): 16 x 64 local tiles, RA in {1, 2, 4}, CA in {1, 2}, 1..32 tokens.
//
// Four local tiles stacked along M form one 64 x 64 super-tile of the balanced
// partition.  A chunk of super-tiles arrives with one bulk copy per sub-band
// and array (union masks, row permutations, value runs: each contiguous along
// the sub-band), and each local tile is decoded straight into the rows of the
// dense tile that its permutation names, so the multiply and the epilogue are
// those of plain tiles.  Other IE-BME shapes take the generic kernel.
#include "us_w4a4_sk.cuh"

namespace us {

bool w4a4_sk_ie_supported(int M, int K, int TM, int TK, int RA, int CA, int N) {
    if (TM != kIeLocalRows || TK != kTK || M % kTM || K % kTK) return false;
    if (!(RA == 1 || RA == 2 || RA == 4) || !(CA == 1 || CA == 2) || RA * CA > 4) return false;
    SkPlan pl;
    return sk_plan(M / kTM, K / kTK, N, false, pl, true) && sk_plan(M / kTM, K / kTK, N, true, pl, true);
}

size_t w4a4_sk_ie_ws(int M, int K, int N) {
    SkPlan pl;
    if (!sk_plan(M / kTM, K / kTK, N, false, pl, true)) return 0;
    return (size_t)pl.G * ntok_for(N, pl.NT) * kTM * 8;   // one posted partial per CTA
}

// p.nTM: 64-row bands; p.ie_ra, p.ie_ca, p.perm as in us_bitmap_ie.  p.ws as
// for launch_w4a4_sk.
us_status launch_w4a4_sk_ie(UsKParams p, cudaStream_t st) {
    SkPlan pl;
    if (!sk_plan(p.nTM, p.nTK, p.N, (p.flags & US_BITMAP_STATIC) != 0, pl, true)) return US_ERR_UNSUPPORTED;
    switch (pl.NT) {
        case 1: return launch_sk_n<8, 1, true>(p, pl, st);
        case 2: return launch_sk_n<16, 2, true>(p, pl, st);
        case 4: return launch_sk_n<32, 4, true>(p, pl, st);
        default: break;
    }
    switch (p.N) {
        case 1: return launch_sk_n<1, 0, true>(p, pl, st);
        case 2: return launch_sk_n<2, 0, true>(p, pl, st);
        case 3: return launch_sk_n<3, 0, true>(p, pl, st);
        case 4: return launch_sk_n<4, 0, true>(p, pl, st);
        case 5: return launch_sk_n<5, 0, true>(p, pl, st);
        case 6: return launch_sk_n<6, 0, true>(p, pl, st);
        case 7: return launch_sk_n<7, 0, true>(p, pl, st);
        case 8: return launch_sk_n<8, 0, true>(p, pl, st);
    }
    return US_ERR_UNSUPPORTED;
}

}  // namespace us
