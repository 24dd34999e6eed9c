// Host-only check of the decode kernels' segment-table bounds test
// (segments_in_block) against the index model that produces the tables
// (build_segments): every table of in-range counters passes, and tables with
// a planted fault (a run past its region, overlapping runs, another head's
// block, a foreign caller row, counters past their capacity) fail.  Built and
// run by test_segment_check_host.py; prints one "name value" line per case.
#include <cstdio>
#include <cstring>
#include <vector>

#include "../compressed_draft_kv_gb300/csrc/masw_internal.cuh"

using namespace masw;

namespace {

constexpr int kRowB = 128;  // D = 64, bf16

struct Fake {
    int L = 2, B = 3, Hkv = 2, S = 4, W = 16, R = 4, M_max = 8, Tmax = 200;
    std::vector<uint8_t> pk, pv, fk, fv, kg, vg;
    DecodeParams p;
    Fake(int mode, int step, int self_attend, int S_ = 4) {
        S = S_;
        std::memset(&p, 0, sizeof(p));
        const int Wc = W + R, C = S + Wc + M_max;
        pk.resize((size_t)L * B * Hkv * C * kRowB);
        pv.resize(pk.size());
        fk.resize((size_t)L * B * Hkv * Tmax * kRowB);
        fv.resize(fk.size());
        kg.resize((size_t)B * Hkv * kRowB);
        vg.resize(kg.size());
        p.pool_k = pk.data();
        p.pool_v = pv.data();
        p.full_k = fk.data();
        p.full_v = fv.data();
        p.k_g = kg.data();
        p.v_g = vg.data();
        p.mode = mode;
        p.B = B;
        p.Hkv = Hkv;
        p.S = S;
        p.W = W;
        p.Wc = Wc;
        p.C = C;
        p.Tmax = Tmax;
        p.M_max = M_max;
        p.self_attend = self_attend;
        p.step = step;
        for (int i = 0; i < MASW_MAX_BATCH / 32; ++i) p.active[i] = step ? 0x5u : 0u;  // rows 0 and 2
    }
    bool check(int lb, int h, int z, int t, int m) const {
        Seg segs[5];
        const int n = build_segments<kRowB>(p, lb, h, z, t, m, segs);
        return segments_in_block<kRowB>(p, lb, h, z, segs, n);
    }
    // every (block, head, row) at every in-range counter pair
    long sweep_failures(int tmax) const {
        long bad = 0;
        for (int lb = 0; lb < L * B; ++lb)
            for (int h = 0; h < Hkv; ++h)
                for (int z = 0; z < B; ++z)
                    for (int t = 0; t <= tmax; ++t)
                        for (int m = 0; m <= M_max; ++m) bad += check(lb, h, z, t, m) ? 0 : 1;
        return bad;
    }
};

void out(const char* name, long v) { std::printf("%s %ld\n", name, v); }

}  // namespace

int main() {
    // 1. tables of in-range counters: no failure (draft, fused step, slot with
    //    self-attention, no sink)
    out("draft_in_range_failures", Fake(kDevModeDraft, 0, 0).sweep_failures(200));
    out("step_in_range_failures", Fake(kDevModeDraft, 1, 0).sweep_failures(199));
    out("slot_in_range_failures", Fake(kDevModeSlot, 0, 1).sweep_failures(200));
    out("nosink_in_range_failures", Fake(kDevModeDraft, 1, 0, 0).sweep_failures(199));
    {
        Fake f(kDevModeFull, 1, 0);
        long bad = 0;
        for (int t = 0; t <= f.Tmax; ++t) bad += f.check(4, 1, 1, t, 0) ? 0 : 1;
        out("full_in_range_failures", bad);
        out("full_t_past_capacity_ok", f.check(4, 1, 1, f.Tmax + 1, 0));
    }
    // 2. counters past their capacity
    {
        Fake f(kDevModeDraft, 0, 0);
        out("slot_count_past_capacity_ok", f.check(1, 0, 0, 150, f.M_max + 1));
        out("slot_count_at_capacity_ok", f.check(1, 0, 0, 150, f.M_max));
    }
    // 3. planted tables
    {
        Fake f(kDevModeDraft, 1, 0);
        Seg segs[6];
        const int n = build_segments<kRowB>(f.p, 3, 1, 2, 105, 5, segs);  // sink, ring (wrapped), slots, new row
        out("reference_table_runs", n);
        out("reference_table_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, segs, n));
        Seg s2[6];
        std::memcpy(s2, segs, sizeof(segs));
        s2[0].len = f.S + 1;  // sink run into the ring
        out("sink_run_into_ring_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n));
        std::memcpy(s2, segs, sizeof(segs));
        s2[n - 2].len = f.M_max + 1;  // slot chain past the block's end
        out("slot_run_past_block_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n));
        std::memcpy(s2, segs, sizeof(segs));
        s2[2] = s2[1];  // the same ring run twice
        out("overlapping_runs_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n));
        std::memcpy(s2, segs, sizeof(segs));
        s2[n - 1].k -= kRowB;  // caller row of another (row, head)
        s2[n - 1].v -= kRowB;
        out("foreign_caller_row_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n));
        std::memcpy(s2, segs, sizeof(segs));
        s2[1].v += kRowB;  // V run not beside its K run
        out("v_offset_mismatch_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n));
        std::memcpy(s2, segs, sizeof(segs));
        s2[0].len = 0;  // empty run
        out("empty_run_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n));
        // the same table checked as another head's: every pool run is outside
        out("other_heads_block_ok", segments_in_block<kRowB>(f.p, 3, 0, 2, segs, n));
        std::memcpy(s2, segs, sizeof(segs));
        s2[n] = s2[0];
        out("six_runs_ok", segments_in_block<kRowB>(f.p, 3, 1, 2, s2, n + 1));
    }
    // 4. the prefill's interleaved row order against a brute-force construction
    //    (raw tokens in order, slot m appended right after raw token tau_m)
    {
        long rows = 0, bad = 0;
        for (int S : {0, 1, 4, 8, 128})
            for (int W : {1, 3, 16, 128, 1024})
                for (int r : {1, 2, 3, 4, 16, 512})
                    for (int T : {1, 5, 60, 100, 257, 333, 1024, 2100}) {
                        const int M = slot_count(T, S, W, r);
                        int pos = 0;
                        for (int i = 1; i <= T; ++i) {
                            bad += interleaved_row(pos++, S, W, r, M) != i;
                            if (is_boundary(i, S, W, r)) bad += interleaved_row(pos++, S, W, r, M) != -((i - S - W) / r);
                        }
                        bad += pos != T + M;
                        rows += pos;
                    }
        out("interleaved_rows", rows);
        out("interleaved_mismatches", bad);
    }
    return 0;
}
