// us_w4a4_sk.cu -- the balanced W4A4 / W2A4 kernel on plain 64 x 64 tiles:
// support checks, workspace size and the launch for 1..32 tokens.  The kernel
// and its shared-memory plan are in us_w4a4_sk.cuh.
#include "us_w4a4_sk.cuh"

namespace us {

bool w4a4_sk_supported(int TM, int TK, int M, int K, int N) {
    if (TM != kTM || TK != kTK) return false;
    SkPlan pl;
    return sk_plan(M / TM, K / TK, N, false, pl);
}

size_t w4a4_sk_ws(int M, int K, int N) {
    SkPlan pl;
    if (!sk_plan(M / kTM, K / kTK, N, false, pl)) return 0;
    return (size_t)pl.G * ntok_for(N, pl.NT) * kTM * 8;   // one posted partial per CTA
}

int w4a4_sk_variant(int N) { return nt_for_tokens(N); }

// p.ws: the workspace, G x NTOK x 64 posted {value, tag} words, zero before the
// first call and left zero by every call.
us_status launch_w4a4_sk(UsKParams p, cudaStream_t st) {
    SkPlan pl;
    if (!sk_plan(p.nTM, p.nTK, p.N, (p.flags & US_BITMAP_STATIC) != 0, pl)) return US_ERR_UNSUPPORTED;
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
