// CPU walk of the attention kernel's unit schedule, for the test suite.
//
// Includes the library's own source, builds the kernel parameters exactly as
// a launch does (build_plan + fill_schedule), then runs the schedule that
// every CTA of the persistent grid runs (unit_of_round / Schedule::at /
// unit_kv_tiles, the same functions the kernel calls) on the host. Checks
// that every (sequence, token block, head group) unit of the call is visited
// exactly once over the whole grid and that the key tiles visited add up to
// the plan's count. No CUDA call is made, so it runs without a GPU.
//
// stdin, one case per line:
//   causal n_q_heads n_kv_heads kv_begin kv_count sm_count n_seqs len_0 ... len_{n-1}
// stdout, one line per case: "ok <units> <kv_tiles> <grid>" or "FAIL <why>".
#include "../long_causal_gqa_gb300/csrc/h3gqa_api.cu"

#include <cstdio>
#include <map>
#include <tuple>

static void run_case(int causal, int hq, int hkv, int kv_begin, int kv_count, int sms,
                     const std::vector<int32_t> &cu)
{
    const int n = (int)cu.size() - 1;
    const int count = kv_count ? kv_count : hkv - kv_begin;
    HostPlan hp;
    const h3gqa_status st = build_plan(cu.data(), n, hq, hkv, 128, causal != 0, count, &hp);
    if (st != H3GQA_OK) {
        std::printf("FAIL plan status %d\n", (int)st);
        return;
    }
    if (hp.n_units == 0) {
        std::printf("ok 0 0 0\n");
        return;
    }
    FwdParams *prm = new FwdParams;
    std::memset(prm, 0, sizeof(*prm));
    prm->causal = causal;
    const int grid = fill_schedule(hp, kv_begin, sms, prm);
    std::map<std::tuple<int, int, int>, int> seen;   // (seq start, block, group) -> visits
    long long tiles = 0, units = 0;
    for (int cta = 0; cta < grid; ++cta) {
        h3gqa::Schedule w;
        w.init(*prm);
        for (long long r = 0;; ++r) {
            if (h3gqa::unit_of_round(r, grid, cta) >= prm->n_units) break;
            const h3gqa::Unit un = w.at(*prm, r, grid, cta);
            if (un.group < 0 || un.group >= prm->n_groups || un.block < 0 ||
                un.block * prm->unit_tokens >= un.seq_len) {
                std::printf("FAIL bad unit cta %d round %lld: seq_start %d len %d block %d group %d\n",
                            cta, r, un.seq_start, un.seq_len, un.block, un.group);
                delete prm;
                return;
            }
            ++seen[std::make_tuple(un.seq_start, un.block, un.group)];
            tiles += h3gqa::unit_kv_tiles(*prm, un);
            ++units;
        }
    }
    long long expected = 0;
    for (int b = 0; b < n; ++b) {
        const int len = cu[b + 1] - cu[b];
        if (len == 0) continue;
        for (int blk = 0; blk * prm->unit_tokens < len; ++blk)
            for (int g = 0; g < prm->n_groups; ++g) {
                ++expected;
                auto it = seen.find(std::make_tuple(cu[b], blk, g));
                if (it == seen.end() || it->second != 1) {
                    std::printf("FAIL unit (seq %d, block %d, group %d) visited %d times\n", b,
                                blk, g, it == seen.end() ? 0 : it->second);
                    delete prm;
                    return;
                }
            }
    }
    if (units != expected || units != hp.n_units || tiles != hp.n_kv_tiles) {
        std::printf("FAIL counts: walked %lld units / %lld tiles, plan %lld / %lld, expected %lld\n",
                    units, tiles, hp.n_units, hp.n_kv_tiles, expected);
    } else {
        std::printf("ok %lld %lld %d\n", units, tiles, grid);
    }
    delete prm;
}

int main()
{
    int causal, hq, hkv, kb, kc, sms, n;
    while (std::scanf("%d %d %d %d %d %d %d", &causal, &hq, &hkv, &kb, &kc, &sms, &n) == 7) {
        std::vector<int32_t> cu(1, 0);
        for (int i = 0; i < n; ++i) {
            int len = 0;
            if (std::scanf("%d", &len) != 1) return 2;
            cu.push_back(cu.back() + len);
        }
        run_case(causal, hq, hkv, kb, kc, sms, cu);
        std::fflush(stdout);
    }
    return 0;
}
