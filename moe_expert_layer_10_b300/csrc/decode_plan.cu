// Host-side planning of the fused decode launch (decode_fused.cu): the K splits of a wave and
// the assignment of its units to CTAs. Both depend only on the wave's routed set, and the CTA a
// unit runs on does not change its result, so outputs stay repeatable bitwise.
#include <algorithm>
#include <vector>

#include "kernels.cuh"
#include "moe.h"

namespace moe {
namespace {

constexpr int BK = 64;                 // K columns per stage of the decode kernels
constexpr int A_BYTES = 128 * BK * 2;  // weight bytes per stage (128 rows of bf16)

}  // namespace

void decode_fused_choose_split(const int* chunk_tok, int n_chunks, int H, int I, int num_sms, int* S_gu_out,
                               int* S_d_out) {
    // load of a unit in bytes: its weights (16 KB per 64-column stage), its token tiles, a
    // fixed cost for the unit's hand-offs, and for a split the partial tile written and read
    const int R_gu = I / 64, R_d = H / 128, KB_gu = H / BK, KB_d = I / BK;
    const double kUnitFixed = 8192.0;
    int best_gu = 1, best_d = 1;
    double best = -1.0, unsplit = 0.0;
    std::vector<double> load(num_sms);
    for (int sg = 1; sg <= kDecodeMaxSplit; ++sg) {
        if (KB_gu / sg < 4) break;
        for (int sd = 1; sd <= kDecodeMaxSplit; ++sd) {
            if (KB_d / sd < 4) break;
            long long units = 0;
            for (int c = 0; c < n_chunks; ++c) units += static_cast<long long>(R_gu) * sg + static_cast<long long>(R_d) * sd;
            if ((sg > 1 || sd > 1) && units > kDecodeSplitUnits) continue;
            std::fill(load.begin(), load.end(), 0.0);
            long long g = 0;
            for (int phase = 0; phase < 2; ++phase) {
                const int R = phase == 0 ? R_gu : R_d, S = phase == 0 ? sg : sd, KB = phase == 0 ? KB_gu : KB_d;
                for (int c = 0; c < n_chunks; ++c) {
                    const int ntp = ((chunk_tok[c] + 15) / 16) * 16;
                    for (int t = 0; t < R; ++t)
                        for (int sp = 0; sp < S; ++sp, ++g) {
                            const int kb = (sp + 1) * KB / S - sp * KB / S;
                            double b = kb * (A_BYTES + ntp * BK * 2.0) + kUnitFixed;
                            if (S > 1) b += 2.0 * ntp * 128 * 4;
                            load[g % num_sms] += b;
                        }
                }
            }
            const double mx = *std::max_element(load.begin(), load.end());
            if (sg == 1 && sd == 1) unsplit = mx;
            if (best < 0 || mx < best * (1.0 - 1e-9)) {
                best = mx;
                best_gu = sg;
                best_d = sd;
            }
        }
    }
    // Splits cost more than this model charges (a split's units are smaller, so less of a down
    // unit's weight stream is already in the ring when its h rows arrive, and each split adds an
    // epilogue pass): on the decode layer at batch 1 the unsplit launch measured 52.8 us against
    // 55.2 us for the chosen (1, 3). So a split is taken only if the model predicts 20 % or more.
    if (best > 0.8 * unsplit) {
        best_gu = 1;
        best_d = 1;
    }
    *S_gu_out = best_gu;
    *S_d_out = best_d;
}

int decode_fused_schedule(int units_gu, int units_d, int kb_gu, int kb_d, int grid, int* sched, int cap) {
    const int n_total = units_gu + units_d;
    // keep, pool_off and at most one moved unit per CTA must fit
    if (grid < 1 || n_total < grid || kb_gu < 1 || kb_d < 1 || 4 * grid + 1 > cap) return 0;
    // Under the round robin CTA b holds units b, b + grid, ...: q + 1 of them for b < r, of which
    // qg + 1 gate/up units for b < rg. So the CTAs form (at most) three index ranges of equal load.
    const int q = n_total / grid, r = n_total % grid, qg = units_gu / grid, rg = units_gu % grid;
    struct Range {
        int b0, b1, count, load;
    };
    const int c0 = std::min(r, rg), c1 = std::max(r, rg);
    Range rs[3] = {{0, c0, q + 1, 0}, {c0, c1, r > rg ? q + 1 : q, 0}, {c1, grid, q, 0}};
    int max_load = 0;
    for (Range& x : rs) {
        const int n_gu = x.b0 < rg ? qg + 1 : qg;
        x.load = n_gu * kb_gu + (x.count - n_gu) * kb_d;
        if (x.b1 > x.b0) max_load = std::max(max_load, x.load);
    }
    // One level of moves: every CTA at the largest load gives its last unit (a down unit of the
    // round robin's last round, so it still runs late, when its h rows exist) to CTAs that stay
    // below that load. Without room for all of them the largest load cannot come down.
    int n_give = 0, room = 0;
    for (const Range& x : rs) {
        if (x.b1 <= x.b0) continue;
        if (x.load == max_load) {
            if (x.count == 0 || x.b0 + (x.count - 1) * grid < units_gu) return 0;  // a gate/up unit last
            n_give += x.b1 - x.b0;
        } else {
            room += (x.b1 - x.b0) * std::max(0, (max_load - 1 - x.load) / kb_d);
        }
    }
    if (n_give == 0 || room < n_give) return 0;
    // the receivers water-filled: the lowest level T at which they hold every moved unit
    auto per = [&](const Range& x, int T) { return x.load < max_load ? std::max(0, (T - x.load) / kb_d) : 0; };
    auto held = [&](int T) {
        int n = 0;
        for (const Range& x : rs)
            if (x.b1 > x.b0) n += (x.b1 - x.b0) * per(x, T);
        return n;
    };
    int lo = 0, hi = max_load - 1;
    while (lo < hi) {
        const int mid = lo + (hi - lo) / 2;
        if (held(mid) >= n_give) hi = mid;
        else lo = mid + 1;
    }
    // per-CTA take: the level's count, less the excess, taken back from the CTAs ending
    // highest (highest index first)
    int take_of[3];
    for (int k = 0; k < 3; ++k) take_of[k] = per(rs[k], lo);
    int excess = held(lo) - n_give;
    int* pool_off = sched + grid;
    int* pool = sched + 2 * grid + 1;
    int drop[3] = {0, 0, 0};  // CTAs of each range (the highest indices) that take one unit fewer
    while (excess > 0) {
        int best = -1;
        for (int k = 0; k < 3; ++k) {
            const int avail = rs[k].b1 - rs[k].b0 - drop[k];
            if (avail > 0 && take_of[k] > 0 &&
                (best < 0 || rs[k].load + take_of[k] * kb_d > rs[best].load + take_of[best] * kb_d))
                best = k;
        }
        if (best < 0) return 0;
        const int n = std::min(excess, rs[best].b1 - rs[best].b0 - drop[best]);
        drop[best] += n;
        excess -= n;
    }
    // write keep[grid], the moved units (givers in CTA order), and pool_off[grid + 1]: receiver
    // b runs the next take units of the pool
    int np = 0;
    for (const Range& x : rs)
        for (int b = x.b0; b < x.b1; ++b) {
            sched[b] = x.load == max_load ? x.count - 1 : x.count;
            if (x.load == max_load) pool[np++] = b + (x.count - 1) * grid;
        }
    int off = 0;
    for (int k = 0; k < 3; ++k)
        for (int b = rs[k].b0; b < rs[k].b1; ++b) {
            pool_off[b] = off;
            off += take_of[k] - (b >= rs[k].b1 - drop[k] ? 1 : 0);
        }
    pool_off[grid] = off;
    if (off != np) return 0;
    return np == n_give ? 3 * grid + 1 + np : 0;
}

}  // namespace moe

int moe_fused_schedule(int units_gu, int units_d, int kb_gu, int kb_d, int grid, int32_t* sched, int cap) {
    if (!sched || units_gu < 0 || units_d < 0 || kb_gu < 1 || kb_d < 1 || grid < 1 || cap < 0) return MOE_E_INVAL;
    return moe::decode_fused_schedule(units_gu, units_d, kb_gu, kb_d, grid, sched, cap);
}
