#include "split_plan.h"

#include <algorithm>
#include <vector>

#include "kda.h"

namespace kda {

constexpr int64_t kWaveBytes = (int64_t)384 << 20;

bool split_applies(int32_t d, int32_t dtype) { return dtype == KDA_BF16 && d == 128; }

int32_t chunks_of(int64_t start, int64_t len) {
    return len > 0 ? (int32_t)((start + len - 1) / kChunk - start / kChunk + 1) : 0;
}

void make_split_plan(int32_t H, int32_t nseq, const int32_t *cu, const int64_t *start, SplitPlan &pl) {
    std::vector<int32_t> nch((size_t)nseq);
    int32_t maxc = 0, nact = 0;
    for (int32_t s = 0; s < nseq; ++s) {
        nch[s] = chunks_of(start[s], (int64_t)cu[s + 1] - cu[s]);
        maxc = std::max(maxc, nch[s]);
        nact += nch[s] > 0;
    }
    pl = SplitPlan();
    if (maxc == 0) return;
    const int64_t per_chunk = (int64_t)nact * H * kImageBytes;
    const int64_t cw_max = std::max<int64_t>(1, kWaveBytes / per_chunk);
    const int64_t nw = (maxc + cw_max - 1) / cw_max;
    const int64_t cw = (maxc + nw - 1) / nw;
    pl.cw = (int32_t)cw;
    pl.nwaves = (int32_t)((maxc + cw - 1) / cw);
    pl.wave_seq_off.assign((size_t)pl.nwaves * nseq, -1);
    for (int32_t w = 0; w < pl.nwaves; ++w) {
        const int32_t b = (int32_t)pl.items.size();
        pl.wave_begin.push_back(b);
        for (int32_t s = 0; s < nseq; ++s) {
            const int32_t l0 = w * pl.cw, l1 = std::min(nch[s], l0 + pl.cw);
            if (l0 >= l1) continue;
            pl.wave_seq_off[(size_t)w * nseq + s] = (int32_t)pl.items.size() - b;
            for (int32_t lc = l0; lc < l1; ++lc) pl.items.push_back(SplitItem{s, lc});
        }
        pl.slot_items = std::max<int64_t>(pl.slot_items, (int64_t)pl.items.size() - b);
    }
    pl.wave_begin.push_back((int32_t)pl.items.size());
}

}  // namespace kda
