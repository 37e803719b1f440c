#include "split_plan.h"

#include <algorithm>
#include <cmath>
#include <vector>

#include "kda.h"

namespace kda {

// Cap on one wave's operand images (one of two workspace slots): 512 MiB while every chain of
// a wave has an SM of its own, 2 GiB when there are more chains than SMs.  Then the chains of a
// wave run in several rounds and every extra wave repeats each round's launch and state
// hand-off, so fewer, larger waves pay (varlen resume, 1024 chains: 65 waves -> 18, 7.15 ms ->
// 5.84 ms); with few chains, smaller waves let them start sooner (no gain measured from larger
// ones for 32 or 64 chains).
constexpr int64_t kWaveBytes = (int64_t)512 << 20, kWaveBytesManyChains = (int64_t)2048 << 20;

bool split_applies(int32_t d, int32_t dtype) { return dtype == KDA_BF16 && d == 128; }

int32_t chunks_of(int64_t start, int64_t len) {
    return len > 0 ? (int32_t)((start + len - 1) / kChunk - start / kChunk + 1) : 0;
}

namespace {

// Cost model of the waves of the split prefill on a GB300 (152 SMs), bf16, d = 128, from
// measurements of the two kernels:
//   chunk prep   ~5.9 us of one SM per (chunk, head) unit (three units in flight per SM, each
//                ~15 us from its first load to its last store);
//   chain        ~2.3 us per chunk on one SM, plus ~4 us to load and hand on its state;
//   launch       ~5 us between the end of one wave's chains and the next.
// While chains run, the next wave's prep uses the SMs the chains leave free, at ~63 % of its
// rate alone (the two compete for HBM: the chains stream operand images, the prep writes them).
// The plan only decides speed, never results: any wave split computes the same outputs.
constexpr double kSMs = 152, kPrepUnitSmUs = 5.9, kPrepUnitLatUs = 15, kChainChunkUs = 2.3,
                 kChainFixedUs = 4, kLaunchUs = 5, kShareEff = 0.63;

// Chunk counts of the sequences, ascending, with prefix sums: the per-wave quantities of a
// candidate split in O(log nseq) each.
struct ChunkHist {
    std::vector<int64_t> n;     // ascending
    std::vector<int64_t> pre;   // pre[i] = n[0] + ... + n[i - 1]
    int64_t H;

    int64_t first_above(int64_t x) const {   // index of the first count > x
        return std::upper_bound(n.begin(), n.end(), x) - n.begin();
    }
    // (chunk, sequence) pairs with local chunk index in [b0, b1)
    int64_t chunks_in(int64_t b0, int64_t b1) const {
        const int64_t i0 = first_above(b0), i1 = first_above(b1 - 1);
        // sequences i0 .. i1-1 end inside the range, i1 .. end cover all of it
        return (pre[i1] - pre[i0]) - (i1 - i0) * b0 + ((int64_t)n.size() - i1) * (b1 - b0);
    }
    int64_t chains_in(int64_t b0) const { return ((int64_t)n.size() - first_above(b0)) * H; }
};

double model_us(const ChunkHist &hs, const std::vector<int32_t> &b) {
    const int W = (int)b.size() - 1;
    const int64_t maxc = hs.n.back();
    double t = 0;
    for (int w = 0; w <= W; ++w) {
        double tc = 0, free_sm = kSMs;
        if (w >= 1) {
            const int64_t b0 = b[w - 1], b1 = std::min<int64_t>(b[w], maxc);
            const int64_t chains = hs.chains_in(b0);
            if (chains > 0) {
                const double rounds = std::ceil((double)chains / kSMs);
                tc = rounds * (kChainFixedUs + kChainChunkUs * (double)(b1 - b0));
                free_sm = chains >= kSMs ? 0 : kSMs - (double)chains;
            }
        }
        double step = tc;
        if (w < W) {
            const double units = (double)hs.chunks_in(b[w], b[w + 1]) * (double)hs.H;
            const double work = units * kPrepUnitSmUs, during = free_sm * tc * kShareEff;
            if (work > during) step = tc + std::max((work - during) / kSMs, w == 0 ? kPrepUnitLatUs : 0.0);
        }
        t += step + kLaunchUs;
    }
    return t;
}

// Wave bounds with sizes proportional to r^w (w = 0 .. W-1), at least one chunk each.
bool geometric_bounds(int64_t maxc, int W, double r, std::vector<int32_t> &b) {
    if (W > maxc) return false;
    std::vector<double> wgt((size_t)W);
    double sum = 0;
    for (int w = 0; w < W; ++w) sum += (wgt[w] = std::pow(r, (double)w));
    b.assign((size_t)W + 1, 0);
    double acc = 0;
    for (int w = 0; w < W; ++w) {
        acc += wgt[w];
        int64_t x = (int64_t)std::llround(acc / sum * (double)maxc);
        x = std::max<int64_t>(x, b[w] + 1);             // at least one chunk
        x = std::min<int64_t>(x, maxc - (W - 1 - w));   // room for the waves after it
        b[w + 1] = (int32_t)x;
    }
    b[W] = (int32_t)maxc;
    return true;
}

}  // namespace

void make_split_plan(int32_t H, int32_t nseq, const int32_t *cu, const int64_t *start, SplitPlan &pl) {
    std::vector<int32_t> nch((size_t)nseq);
    ChunkHist hs;
    hs.H = H;
    int32_t maxc = 0;
    for (int32_t s = 0; s < nseq; ++s) {
        nch[s] = chunks_of(start[s], (int64_t)cu[s + 1] - cu[s]);
        maxc = std::max(maxc, nch[s]);
        if (nch[s] > 0) hs.n.push_back(nch[s]);
    }
    pl = SplitPlan();
    if (maxc == 0) return;
    std::sort(hs.n.begin(), hs.n.end());
    hs.pre.assign(hs.n.size() + 1, 0);
    for (size_t i = 0; i < hs.n.size(); ++i) hs.pre[i + 1] = hs.pre[i] + hs.n[i];

    // Fewest waves whose images fit a slot if every wave were equal; candidates from there up
    // to six more waves, sizes geometric in the wave index (decreasing when chunk preparation
    // dominates, increasing when the chains do); the modelled fastest split that keeps every
    // slot under the cap wins.  The equal split is always a candidate.
    const int64_t unit_bytes = (int64_t)H * kImageBytes;
    const int64_t per_chunk = (int64_t)hs.n.size() * unit_bytes;
    const int64_t wave_bytes = (int64_t)hs.n.size() * H > (int64_t)kSMs ? kWaveBytesManyChains : kWaveBytes;
    const int64_t cw_max = std::max<int64_t>(1, wave_bytes / per_chunk);
    const int W0 = (int)((maxc + cw_max - 1) / cw_max);
    auto fits = [&](const std::vector<int32_t> &b) {
        for (size_t w = 0; w + 1 < b.size(); ++w)
            if (b[w + 1] <= b[w] || hs.chunks_in(b[w], b[w + 1]) * unit_bytes > wave_bytes) return false;
        return true;
    };
    std::vector<int32_t> best, cand;
    double best_t = 0;
    for (int W = W0; W <= W0 + 6 && W <= maxc; ++W)
        for (int ri = -12; ri <= 12; ++ri) {
            const double r = std::pow(2.0, ri / 8.0);   // 0.35 .. 2.8
            if (!geometric_bounds(maxc, W, r, cand) || !fits(cand)) continue;
            const double t = model_us(hs, cand);
            if (best.empty() || t < best_t) {
                best = cand;
                best_t = t;
            }
        }
    if (best.empty()) {   // equal waves of cw_max chunks always fit
        for (int64_t x = 0; x < maxc; x += cw_max) best.push_back((int32_t)x);
        best.push_back(maxc);
    }

    pl.wave_c0 = best;
    pl.nwaves = (int32_t)best.size() - 1;
    pl.wave_seq_off.assign((size_t)pl.nwaves * nseq, -1);
    for (int32_t w = 0; w < pl.nwaves; ++w) {
        const int32_t b = (int32_t)pl.items.size();
        pl.wave_begin.push_back(b);
        for (int32_t s = 0; s < nseq; ++s) {
            const int32_t l0 = pl.wave_c0[w], l1 = std::min(nch[s], pl.wave_c0[w + 1]);
            if (l0 >= l1) continue;
            pl.wave_seq_off[(size_t)w * nseq + s] = (int32_t)pl.items.size() - b;
            for (int32_t lc = l0; lc < l1; ++lc)
                pl.items.push_back(SplitItem{s, lc, (int32_t)(cu[s] + (start[s] / kChunk + lc) * kChunk - start[s]), -1});
        }
        pl.slot_items = std::max<int64_t>(pl.slot_items, (int64_t)pl.items.size() - b);
    }
    pl.wave_begin.push_back((int32_t)pl.items.size());
}

}  // namespace kda
