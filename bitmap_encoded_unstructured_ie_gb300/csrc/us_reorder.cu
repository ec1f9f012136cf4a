// us_reorder.cu -- bitmap-aware row reordering for IE-BME with areas (host,
// offline).
//
// "UnionSparse: An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM
// Inference on Edge", section V-B: the rows of a local tile are partitioned
// into groups of RA (one row from each row partition); a group activates, at
// grouped column j, the OR of its rows' nonzero flags over the CA column
// partitions (Eq. 3), and costs the number of such active grouped columns
// (Eq. 4).  The partition of minimum total cost is found exactly by dynamic
// programming over row subsets whose smallest row is always grouped first
// (Eq. 5, Algorithm 1), then canonicalised (rows ascending inside a group,
// groups lexicographic) and laid out partition-wise: row p*(HL/RA) + g of the
// reordered tile is row p of group g.
//
// The pages run this once, offline, on the CPU; so does this library.  Here
// the subsets are visited bottom-up in increasing numeric order (removing a
// group only lowers the subset's value), and every group's cost comes from a
// table over row sets built from per-row activity bitsets.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "us_internal.h"

namespace {

struct Bits128 {
    uint64_t lo = 0, hi = 0;
};

// Minimum-cost grouping of one tile; perm receives HL row indices.
bool reorder_tile(const std::vector<Bits128>& act, int HL, int RA, uint8_t* perm, std::vector<int32_t>& F,
                  std::vector<uint32_t>& best, std::vector<int16_t>& gcost) {
    const uint32_t nS = 1u << HL;
    // cost of every row set of size RA: active grouped columns of the union
    for (uint32_t g = 0; g < nS; ++g) {
        if (__builtin_popcount(g) != RA) continue;
        Bits128 u;
        for (int r = 0; r < HL; ++r)
            if ((g >> r) & 1u) { u.lo |= act[r].lo; u.hi |= act[r].hi; }
        gcost[g] = (int16_t)(__builtin_popcountll(u.lo) + __builtin_popcountll(u.hi));
    }
    const int32_t kInf = INT32_MAX;
    F[0] = 0;
    for (uint32_t S = 1; S < nS; ++S) {
        F[S] = kInf;
        if (__builtin_popcount(S) % RA) continue;
        const uint32_t low = S & (~S + 1u);              // the smallest row must join a group now
        uint32_t rest = S & ~low;
        int rows[32], nr = 0;
        while (rest) {
            rows[nr++] = __builtin_ctz(rest);
            rest &= rest - 1u;
        }
        // every way to pick the RA - 1 partners from the other rows of S
        auto consider = [&](uint32_t g) {
            const int32_t sub = F[S & ~g];
            if (sub != kInf && sub + gcost[g] < F[S]) {
                F[S] = sub + gcost[g];
                best[S] = g;
            }
        };
        if (RA == 1) {
            consider(low);
        } else if (RA == 2) {
            for (int a = 0; a < nr; ++a) consider(low | 1u << rows[a]);
        } else if (RA == 3) {
            for (int a = 0; a < nr; ++a)
                for (int b = a + 1; b < nr; ++b) consider(low | 1u << rows[a] | 1u << rows[b]);
        } else {
            for (int a = 0; a < nr; ++a)
                for (int b = a + 1; b < nr; ++b)
                    for (int c = b + 1; c < nr; ++c) consider(low | 1u << rows[a] | 1u << rows[b] | 1u << rows[c]);
        }
    }
    // groups of the optimum; each is ascending as a bit set; ordering the groups
    // by their smallest row is the lexicographic order of disjoint groups
    std::vector<uint32_t> groups;
    for (uint32_t S = nS - 1; S;) {
        groups.push_back(best[S]);
        S &= ~best[S];
    }
    std::sort(groups.begin(), groups.end(),
              [](uint32_t a, uint32_t b) { return __builtin_ctz(a) < __builtin_ctz(b); });
    const int G = HL / RA;
    for (int g = 0; g < G; ++g) {
        uint32_t bits = groups[g];
        for (int p = 0; p < RA; ++p) {
            const int r = __builtin_ctz(bits);
            bits &= bits - 1u;
            perm[p * G + g] = (uint8_t)r;
        }
    }
    return true;
}

}  // namespace

extern "C" {

us_status us_reorder_rows(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, us_elem elem,
                          uint8_t* perm, int nthreads) {
    if (!W || !perm || M <= 0 || K <= 0 || TM <= 0 || TK <= 0 || ldw < K) return US_ERR_INVALID_ARG;
    if (RA < 1 || RA > 4 || CA < 1 || CA > 4 || TM % RA || TK % CA || M % TM || K % TK) return US_ERR_INVALID_ARG;
    if (elem != US_F16 && elem != US_I4) return US_ERR_INVALID_ARG;
    if (TM > 20 || TK / CA > 128) return US_ERR_UNSUPPORTED;      // the exact DP is exponential in TM
    const int nTM = M / TM, nTK = K / TK, LK = TK / CA;
    const int64_t nT = (int64_t)nTM * nTK;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    auto work = [&](int tid) {
        std::vector<int32_t> F((size_t)1 << TM);
        std::vector<uint32_t> best((size_t)1 << TM, 0u);
        std::vector<int16_t> gcost((size_t)1 << TM, 0);
        std::vector<Bits128> act(TM);
        for (int64_t t = tid; t < nT; t += nthreads) {
            const int tm = (int)(t / nTK), tk = (int)(t % nTK);
            for (int r = 0; r < TM; ++r) {
                Bits128 b;
                const int64_t row = (int64_t)(tm * TM + r) * ldw + (int64_t)tk * TK;
                for (int c = 0; c < CA; ++c)
                    for (int j = 0; j < LK; ++j) {
                        const int64_t idx = row + c * LK + j;
                        const bool nz = elem == US_F16 ? (static_cast<const uint16_t*>(W)[idx] & 0x7FFFu) != 0
                                                       : static_cast<const int8_t*>(W)[idx] != 0;
                        if (nz) {
                            if (j < 64) b.lo |= 1ull << j;
                            else b.hi |= 1ull << (j - 64);
                        }
                    }
                act[r] = b;
            }
            reorder_tile(act, TM, RA, perm + t * TM, F, best, gcost);
        }
    };
    std::vector<std::thread> pool;
    for (int i = 1; i < nthreads; ++i) pool.emplace_back(work, i);
    work(0);
    for (auto& th : pool) th.join();
    return US_OK;
}

}  // extern "C"
