// Causal GQA prefill forward for sm_103a: TMA-staged Q/K/V tiles, tcgen05
// MMAs into tensor memory, fp32 online softmax in exp2 form, per-row LSE.
//
// The step is the causal grouped-query attention of antirez/h3.c issue #47
// ("Qwen layer 0 causal GQA failed: causal attention sequence 10231 exceeds
// threadgroup memory", "Error"). That issue's kernel keeps the whole fp32
// score row on chip, which caps the sequence near 7700 tokens; its
// "Suggested fix directions" propose tiling the score row. Here the score
// row is never materialised: keys stream through 128-key tiles and the
// softmax is carried online (running max, running sum, rescaled output), so
// on-chip state per query row is O(tile) and there is no length bound.
//
// Work decomposition ("pack-GQA"): a query tile is 128 MMA rows made of the
// query heads of one head group times consecutive tokens. A head group is
// `tile_heads` query heads that read the same KV head: all G = Hq/Hkv of them
// when G <= 128 (more generally the largest divisor of G that is <= 128, so a
// KV head with G > 128 heads has G/tile_heads groups). A tile holds
// tile_tokens = floor(128 / tile_heads) tokens (row r = head r / tile_tokens
// of the group, token r % tile_tokens); rows past tile_heads * tile_tokens
// are unused. A unit is two such tiles (2 * tile_tokens consecutive tokens)
// plus every 128-key tile up to its last token, so each K/V tile staged in
// shared memory feeds every query head of the group.
//
// CTA roles (352 threads, one CTA per SM, persistent over units):
//   warps 0-3  softmax for query tile 0 (thread = MMA row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer (one lane)
//   warp  9    TMEM allocator; MMA issuer for query tile 0 (one lane)
//   warp 10    MMA issuer for query tile 1 (one lane)
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512);
// P (bf16, two per column) overwrites the first 64 columns of its S.
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx_sm103a.cuh"

namespace h3gqa {

// The unit schedule below also compiles as host code, so that it can be
// walked on the CPU.
#define H3GQA_HD __host__ __device__ __forceinline__

H3GQA_HD int imin(int a, int b) { return a < b ? a : b; }

constexpr int kHeadDim = 128;
constexpr int kRows = 128;                 // MMA M: query rows per tile
constexpr int kKeys = 128;                 // keys per K/V tile
constexpr int kStages = 4;                 // K/V ring depth (K and V take one stage each)
constexpr int kMaxSeqs = 1024;
constexpr int kThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kSubTileBytes = 128 * 128;          // 128 rows x 64 bf16 (one 128-B swizzle span)
constexpr uint32_t kTileBytes = 2 * kSubTileBytes;     // 128 rows x 128 bf16
constexpr uint32_t kQOff = 0;                          // two query tiles
constexpr uint32_t kKvOff = kQOff + 2 * kTileBytes;
constexpr uint32_t kRopeOff = kKvOff + kStages * kTileBytes;   // cos rows, then sin rows, of one unit
constexpr int kRopeMaxTokens = 32;                             // staged when a unit has <= 32 tokens (G >= 8)
// Each table's 32 rows of 64 fp32 come in as two TMA boxes of 32 rows x 32
// floats (128 bytes) in the 128-byte-swizzled layout, so the eight tokens a
// quarter-warp reads at one column fall in eight different bank groups.
constexpr uint32_t kRopeHalfBytes = kRopeMaxTokens * 128;      // one box
constexpr uint32_t kRopeBytes = 2 * 2 * kRopeHalfBytes;        // cos, sin x two halves
constexpr uint32_t kBarOff = kRopeOff + kRopeBytes;
// barrier slots
constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarKvFull = 2, kBarKvEmpty = 2 + kStages,
              kBarSFull = 2 + 2 * kStages, kBarPFull = kBarSFull + 2, kBarOFull = kBarPFull + 2,
              kBarDrain = kBarOFull + 2, kBarQReady = kBarDrain + 2, kNumBars = kBarQReady + 2;
constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;  // [0] TMEM base, [1] abort flag, [2..3] MMA turn counters
constexpr uint32_t kSchedOff = kMiscOff + 16;          // softmax threads' unit-schedule state, one slot each
constexpr uint32_t kSchedSlotBytes = 24;
constexpr uint32_t kQNormWOff = kSchedOff + 256 * kSchedSlotBytes;   // the Q norm weight, bf16 [128]
constexpr uint32_t kSmemBytes = kQNormWOff + kHeadDim * 2 + 1024;     // + slack to align the base to 1024
// TMA destinations with the 128-byte swizzle need 1024-byte alignment; the
// norm weight is read as 16-byte vectors, barriers and schedule slots as
// 8-byte words
static_assert(kQOff % 1024 == 0 && kKvOff % 1024 == 0 && kRopeOff % 1024 == 0, "TMA tile alignment");
static_assert(kBarOff % 8 == 0 && kSchedOff % 8 == 0 && kQNormWOff % 16 == 0, "shared-memory field alignment");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only if the max grew by > 2^8
#ifndef H3GQA_WAIT_NS
#define H3GQA_WAIT_NS 2000000000ull
#endif
constexpr uint64_t kWaitNs = H3GQA_WAIT_NS;         // wall time before a pipeline wait gives up

constexpr uint64_t kDrainNs = 2000000000ull;        // wall time allowed for in-flight copies to land

// Device-side timeout record (per device, static): bit 0 producer, bit 1
// MMA issuer, bit 2 softmax, bit 3 teardown drain.
__device__ unsigned int g_timeout_flags;

struct FwdParams {
    CUtensorMap map_q;      // q [Hq][T][128], box {64, tile_tokens, tile_heads}
    CUtensorMap map_k;      // k [Hkv][T][128], box {64, 128, 1}
    CUtensorMap map_v;      // v [Hkv][T][128], box {64, 128, 1}
    CUtensorMap map_cos;    // rotary cos [T][64] fp32, box {32, 32} (staged rotary only)
    CUtensorMap map_sin;    // rotary sin, likewise
    void *o;                // bf16 (or int8 codes) [Hq][T][128] or [T][Hq][128]
    float *lse;             // fp32 [Hq][T]
    float *o_scale;         // int8 output only: one fp32 scale per (token, head) row
    unsigned int *status;   // optional per-call word: timeout bits are ORed into it
    int causal;             // 1: key j visible to query i iff j <= i; 0: all keys of the sequence
    int out_token_major;    // 0: o is [Hq][T][128]; 1: o is [T][Hq][128] (o_scale likewise)
    int out_int8;           // 0: bf16 o; 1: int8 codes, o ~= code * o_scale
    int o_align32;          // o's base is 32-byte aligned (every row then is too)
    int n_q_heads;
    // Q prologue (RMS-norm and/or rotary embedding applied to each Q tile in
    // shared memory right after it lands): prep_q != 0 enables it.
    int prep_q;
    int stage_rope;             // rotary rows of each unit copied into shared memory with its Q
    const uint16_t *q_norm_w;   // bf16 [128] or null
    const float *rope_cos;      // fp32 [T][64] or null
    const float *rope_sin;
    float norm_eps;
    long long total_tokens;
    long long n_units;
    int n_groups;           // head groups this call covers (a head shard covers a subset)
    int group0;             // first head group of this call
    int groups_per_kv;      // head groups per KV head (G / tile_heads)
    int tile_heads;         // query heads per tile
    int tile_tokens;        // floor(128 / tile_heads) tokens per query tile
    int tile_rows;          // tile_heads * tile_tokens used MMA rows (<= 128)
    int unit_tokens;        // 2 * tile_tokens
    int pow2;               // unit_tokens is a power of two dividing 128: shift paths below
    int unit_tokens_log2;   // pow2 only
    int blocks_per_class;   // pow2 only: 128 / unit_tokens units of one sequence visit the same K/V tiles
    int blocks_per_class_log2;
    int n_seqs;             // non-empty sequences, sorted by length (descending)
    int c_max;              // highest cost class (K/V tiles of the longest sequence's last block)
    int full_windows;       // (n_units / n_groups) / grid: whole windows of the unit schedule
    unsigned int q_tx_bytes;   // bytes of one unit's two Q tiles as TMA writes them
    float scale_log2;       // scale * log2(e)
    int seq_start[kMaxSeqs];
    int seq_len[kMaxSeqs];
};

struct Unit {
    int seq_start;
    int seq_len;
    int block;      // token block index inside the sequence
    int group;      // head group, relative to the call's first group
};

// Walks the global longest-first order of block slots (a slot is one token
// block of one sequence; it becomes a unit once a head group is attached).
// Slots are grouped by cost class c (= K/V tiles up to the block's last
// token, from c_max down to 1); inside a class by sequence (longest first),
// then block. Block k of U tokens reaches tile floor((kU + U - 1) / 128), so
// class c starts at block floor(128 (c - 1) / U); when U divides 128 every
// class holds 128 / U blocks. Without the causal rule every slot of a
// sequence costs the same: longest sequence first, then block. Every role of
// a CTA runs the same walk, so no schedule is stored anywhere. Successive
// seeks must not go backwards.
struct UnitWalker {
    int c;
    int i;
    int base;       // first slot of the current (class, sequence) group; slots fit in int

    H3GQA_HD void init(const FwdParams &p)
    {
        c = p.c_max;
        i = 0;
        base = 0;
    }

    H3GQA_HD int blocks_of(const FwdParams &p, int seq) const
    {
        const int n = p.seq_len[seq] + p.unit_tokens - 1;
        return p.pow2 ? n >> p.unit_tokens_log2 : n / p.unit_tokens;
    }

    // first block of cost class cls (any sequence long enough to have it)
    H3GQA_HD int class_lo(const FwdParams &p, int cls) const
    {
        return p.pow2 ? (cls - 1) << p.blocks_per_class_log2 : (kKeys * (cls - 1)) / p.unit_tokens;
    }

    H3GQA_HD int blocks_in_class(const FwdParams &p, int cls, int seq) const
    {
        const int lo = class_lo(p, cls);
        const int hi = imin(class_lo(p, cls + 1), blocks_of(p, seq));
        return hi > lo ? hi - lo : 0;
    }

    // slot must not decrease from one call to the next, and slot < n_units / n_groups.
    H3GQA_HD Unit seek(const FwdParams &p, int slot)
    {
        Unit r;
        if (p.causal && p.n_seqs == 1) {
            const int nblk = blocks_of(p, 0);
            if (p.pow2) {
                // One sequence: the top class holds the blocks past the last
                // whole class, every lower class blocks_per_class of them.
                const int top = nblk - ((p.c_max - 1) << p.blocks_per_class_log2);
                if (slot < top) {
                    r.block = ((p.c_max - 1) << p.blocks_per_class_log2) + slot;
                } else {
                    const int s2 = slot - top;
                    const int cls = p.c_max - 1 - (s2 >> p.blocks_per_class_log2);
                    r.block = ((cls - 1) << p.blocks_per_class_log2) + (s2 & (p.blocks_per_class - 1));
                }
            } else {
                // block cost grows with the block index: last block first
                r.block = nblk - 1 - slot;
            }
        } else if (!p.causal) {
            for (;;) {
                const int cnt = blocks_of(p, i);
                if (slot < base + cnt) break;
                base += cnt;
                ++i;
            }
            r.block = slot - base;
        } else {
            for (;;) {
                const int cnt = blocks_in_class(p, c, i);
                if (slot < base + cnt) break;
                base += cnt;
                ++i;
                if (i >= p.n_seqs || blocks_in_class(p, c, i) == 0) {
                    i = 0;
                    --c;
                }
            }
            r.block = class_lo(p, c) + (slot - base);
        }
        r.seq_start = p.seq_start[i];
        r.seq_len = p.seq_len[i];
        r.group = 0;
        return r;
    }
};

// Key tiles a unit visits: up to its last token inside the sequence
// (causal), or the whole sequence.
H3GQA_HD int unit_kv_tiles(const FwdParams &p, const Unit &un)
{
    const int last = imin(un.block * p.unit_tokens + p.unit_tokens, un.seq_len) - 1;
    return p.causal ? last / kKeys + 1 : (un.seq_len + kKeys - 1) / kKeys;
}

// Round r of the static schedule hands CTA x the unit index r*grid + x on
// even rounds and r*grid + (grid-1-x) on odd ones (a snake), which evens out
// the falling unit costs of the longest-first order.
H3GQA_HD long long unit_of_round(long long r, int grid, int cta)
{
    const long long g = grid;
    const long long x = cta;
    return r * g + ((r & 1) ? (g - 1 - x) : x);
}

// Maps unit indices to (slot, head group). The slot order is cut into windows
// of grid slots; inside a window the head group is the slowest index, so the
// grid's CTAs, which run one round at a time, work on one group and share its
// K/V tiles in L2 (with the group fastest, a round spans every KV head and a
// long sequence's K/V no longer fits in L2). Round r of window r / n_groups
// runs group r mod n_groups on slot x or grid-1-x; even and odd rounds keep a
// walker each, so both only move forward. The last, partial window keeps the
// group fastest.
struct Schedule {
    UnitWalker even, odd;

    H3GQA_HD void init(const FwdParams &p)
    {
        even.init(p);
        odd.init(p);
    }

    // The unit of round r (r < n_units < 2^31) for CTA `cta` of a grid of
    // `g`; r must not decrease between calls.
    H3GQA_HD Unit at(const FwdParams &p, long long r64, int g, int cta)
    {
        const int r = (int)r64;
        const int x = (r & 1) ? g - 1 - cta : cta;
        const int w = r / p.n_groups;
        Unit un;
        if (w < p.full_windows) {
            un = ((r & 1) ? odd : even).seek(p, w * g + x);
            un.group = r - w * p.n_groups;
        } else {
            const int q = (r - p.full_windows * p.n_groups) * g + x;
            const int qs = q / p.n_groups;
            un = even.seek(p, p.full_windows * g + qs);
            un.group = q - qs * p.n_groups;
        }
        return un;
    }
};
static_assert(sizeof(Schedule) == kSchedSlotBytes, "schedule slot size");

// Raises timeout bit `who` in the device-wide flag and in the call's own
// status word (if it gave one).
__device__ __forceinline__ void report_timeout(unsigned int *status, unsigned int who)
{
    atomicOr(&g_timeout_flags, who);
    if (status != nullptr) atomicOr(status, who);
}

__device__ __forceinline__ bool wait_poll(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned int who, unsigned int *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    // Each failed poll has been suspended up to the capped hint (20 us), so
    // checking the clock and the abort flag on every one costs nothing.
    while (!mbar_try_wait_capped(bar, parity)) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            report_timeout(status, who);
            return false;
        }
    }
    return true;
}

// Waits without giving up early on an abort (teardown: copies or MMAs in
// flight must finish before the CTA releases its memory); bounded in time.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned int *status)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_capped(bar, parity)) {
        if (global_timer_ns() - t0 > kDrainNs) {
            report_timeout(status, 8u);
            return false;
        }
    }
    return true;
}

// All 32 lanes wait; the result is agreed across the warp so that the
// .sync.aligned TMEM instructions after it never run on a partial warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned int who, unsigned int *status)
{
    bool ok = wait_poll(bar, parity, abort_flag, who, status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    return ok;
}

// One instance per output dtype and per Q prologue on/off (p.out_int8 and
// p.prep_q equal the template arguments), so that a launch carries only the
// epilogue and prologue code it runs: the code of a unit boundary, run once
// per unit between the large unrolled softmax blocks, then fetches less.
template <bool kInt8, bool kPrepQ>
__global__ void __launch_bounds__(kThreads, 1)
causal_gqa_fwd_kernel(const __grid_constant__ FwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + kQOff;
    const uint32_t sKV = sbase + kKvOff;
    auto bar = [&](int i) -> uint32_t { return sbase + kBarOff + 8u * (uint32_t)i; };
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem + kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned int *const status = p.status;

    if (kPrepQ && p.q_norm_w != nullptr && threadIdx.x < kHeadDim * 2 / 16) {
        // The Q norm weight is read by every row of every unit's Q tile: one
        // copy in shared memory (global loads would mostly miss the small L1
        // that shared memory leaves and sit on the transform's critical path).
        reinterpret_cast<uint4 *>(smem + kQNormWOff)[threadIdx.x] =
            __ldg(reinterpret_cast<const uint4 *>(p.q_norm_w) + threadIdx.x);
    }
    if (p.tile_rows < kRows) {
        // Query tiles with unused MMA rows: TMA never writes those rows, so
        // they are zeroed once here (their scores stay finite; every MMA row
        // is independent of the others, and unused rows are never stored).
        uint4 *q4 = reinterpret_cast<uint4 *>(smem + kQOff);
        for (int i = threadIdx.x; i < (int)(2 * kTileBytes / 16); i += kThreads)
            q4[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(kBarQFull), 1);
        mbar_init(bar(kBarQEmpty), 2);              // one commit per MMA issuer
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarKvFull + s), 1);
            mbar_init(bar(kBarKvEmpty + s), 2);     // one commit per MMA issuer
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(kBarSFull + t), 1);
            mbar_init(bar(kBarPFull + t), kRows);
            mbar_init(bar(kBarOFull + t), 1);
        }
        mbar_init(bar(kBarQReady), kRows);
        mbar_init(bar(kBarQReady + 1), kRows);
        mbar_init(bar(kBarDrain), 1);
        mbar_init(bar(kBarDrain + 1), 1);
        *abort_flag = 0;
        misc[2] = 0;
        misc[3] = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(const_cast<uint32_t *>(misc)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_map(&p.map_q);
            tma_prefetch_map(&p.map_k);
            tma_prefetch_map(&p.map_v);
            if (p.stage_rope) {
                tma_prefetch_map(&p.map_cos);
                tma_prefetch_map(&p.map_sin);
            }
            Schedule w;
            w.init(p);
            // K/V tiles are read again by every unit of their KV head and
            // cost class: kept in L2 over the streamed Q and O lines (paired
            // runs: +0.4-0.9% without the Q prologue, -1% with it, whose
            // keys the K pass has just written)
            const uint64_t pol_kv = kPrepQ ? 0ull : l2_policy_evict_last();
            uint32_t kv_it = 0, unit_it = 0;
            int last_kv_parity[kStages];
            for (int s = 0; s < kStages; ++s) last_kv_parity[s] = -1;
            int last_q_parity = -1;
            bool ok = true;
            for (long long r = 0; ok; ++r) {
                const long long u = unit_of_round(r, gridDim.x, blockIdx.x);
                if (u >= p.n_units) break;
                const Unit un = w.at(p, r, gridDim.x, blockIdx.x);
                const int tb = un.block * p.unit_tokens;
                const int n_kv = unit_kv_tiles(p, un);
                const int grp = p.group0 + un.group;               // absolute head group
                const int kvh = p.groups_per_kv == 1 ? grp : grp / p.groups_per_kv;
                // K and V of key tile j into the next two ring stages
                auto load_kv = [&](int j) -> bool {
                    for (int kind = 0; kind < 2; ++kind) {
                        const uint32_t s = kv_it % kStages;
                        const uint32_t ph = (kv_it / kStages) & 1;
                        if (!wait_poll(bar(kBarKvEmpty + s), ph ^ 1, abort_flag, 1u, status)) return false;
                        mbar_arrive_expect_tx(bar(kBarKvFull + s), kTileBytes);
                        last_kv_parity[s] = (int)ph;
                        const CUtensorMap *map = kind ? &p.map_v : &p.map_k;
                        for (int h = 0; h < 2; ++h) {
                            if (kPrepQ)
                                tma_load_3d(sKV + s * kTileBytes + (uint32_t)h * kSubTileBytes, map,
                                            bar(kBarKvFull + s), 64 * h, un.seq_start + j * kKeys, kvh);
                            else
                                tma_load_3d_hint(sKV + s * kTileBytes + (uint32_t)h * kSubTileBytes, map,
                                                 bar(kBarKvFull + s), 64 * h, un.seq_start + j * kKeys, kvh,
                                                 pol_kv);
                        }
                        ++kv_it;
                    }
                    return true;
                };
                // The unit's first K/V tile is issued before waiting for the Q
                // buffer, so it is in flight while the last unit finishes.
                if (!load_kv(0)) { ok = false; break; }
                if (!wait_poll(bar(kBarQEmpty), (unit_it & 1) ^ 1, abort_flag, 1u, status)) { ok = false; break; }
                const int tok0 = un.seq_start + tb;
                mbar_arrive_expect_tx(bar(kBarQFull), p.q_tx_bytes + (p.stage_rope ? kRopeBytes : 0u));
                last_q_parity = unit_it & 1;
                if (p.stage_rope) {
                    // the unit's rotary rows: 32 rows of each table (rows past
                    // T read as zero), two 128-byte halves each
                    for (int h = 0; h < 2; ++h) {
                        tma_load_2d(sbase + kRopeOff + (uint32_t)h * kRopeHalfBytes, &p.map_cos, bar(kBarQFull),
                                    32 * h, tok0);
                        tma_load_2d(sbase + kRopeOff + (uint32_t)(2 + h) * kRopeHalfBytes, &p.map_sin,
                                    bar(kBarQFull), 32 * h, tok0);
                    }
                }
                for (int t = 0; t < 2; ++t)
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(sQ + (uint32_t)(t * 2 + h) * kSubTileBytes, &p.map_q,
                                    bar(kBarQFull), 64 * h, un.seq_start + tb + t * p.tile_tokens,
                                    grp * p.tile_heads);
                for (int j = 1; j < n_kv && ok; ++j)
                    if (!load_kv(j)) ok = false;
                if (!ok) break;
                ++unit_it;
            }
            if (!ok) {
                // Let every copy already issued land before the CTA exits.
                for (int s = 0; s < kStages; ++s)
                    if (last_kv_parity[s] >= 0) wait_drain(bar(kBarKvFull + s), (uint32_t)last_kv_parity[s], status);
                if (last_q_parity >= 0) wait_drain(bar(kBarQFull), (uint32_t)last_q_parity, status);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ------------------------------------------------------ MMA issuers
        // One issuing lane per query tile. tcgen05.mma issue stalls while the
        // tensor pipe's queue is full, so a single issuer would leave the
        // pipe idle during its own barrier waits and commits. The two
        // issuers pass a turn token back and forth (tile 0, tile 1, tile 0,
        // ...): the tensor pipe alternates between the tiles (so one tile's
        // softmax overlaps the other tile's MMAs), and each issuer does its
        // bookkeeping while the other one's batch runs.
        if (lane == 0) {
            const int t = warp - kMmaWarp;
            constexpr uint32_t idS = idesc_bf16_f32(kRows, kKeys, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kRows, kHeadDim, true);
            const uint32_t tS = tmem + (uint32_t)t * 128u;
            const uint32_t tO = tmem + 256u + (uint32_t)t * 128u;
            const uint32_t sQt = sQ + (uint32_t)t * kTileBytes;
            Schedule w;
            w.init(p);
            uint32_t kv_it = 0, unit_it = 0, p_phase = 0, turns = 0;
            bool ok = true;
            // Turn k of issuer 0 follows turn k-1 of issuer 1; turn k of
            // issuer 1 follows turn k of issuer 0.
            // The token is a pair of shared-memory counters (a plain volatile
            // spin wakes faster than an mbarrier): issuer t may start its
            // turn k once the other issuer has published `done` >= the
            // count it needs.
            volatile uint32_t *my_flag = misc + 2 + t;          // written by the other issuer
            volatile uint32_t *their_flag = misc + 2 + (t ^ 1);
            auto take_turn = [&]() -> bool {
                const uint32_t need = t == 0 ? turns : turns + 1;   // other's completed turns
                if (need == 0) return true;
                if (*my_flag >= need) return true;
                const uint64_t t0 = global_timer_ns();
                for (uint32_t n = 0; *my_flag < need; ++n) {
                    if ((n & 255u) == 255u) {
                        if (*abort_flag) return false;
                        if (global_timer_ns() - t0 > kWaitNs) {
                            *abort_flag = 1;
                            report_timeout(status, 2u);
                            return false;
                        }
                    }
                }
                return true;
            };
            auto pass_turn = [&]() {
                ++turns;
                *their_flag = turns;
            };

            // Shared-memory descriptors (128-byte swizzle), split in words:
            // Q and K are K-major (8-row groups 1024 B apart; the leading
            // offset is unused), V is the MN-major B operand of P.V (64 head
            // dims per 128-B row, the next 64 dims one 16 KB sub-tile further,
            // 8-key groups 1024 B apart). A stage or k-step is a constant
            // added to the low word of stage 0 / of this tile's Q.
            constexpr uint32_t kHiK = sdesc_hi_sw128(1024);
            constexpr uint32_t kHiV = sdesc_hi_sw128(1024);
            const uint32_t q_lo = sdesc_lo(sQt, 16);
            const uint32_t k_lo0 = sdesc_lo(sKV, 16);
            const uint32_t v_lo0 = sdesc_lo(sKV, kSubTileBytes);
            auto issue_s = [&](uint32_t stage) {
                const uint32_t k_lo = k_lo0 + stage * (kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t off = ((uint32_t)(kk >> 2) * kSubTileBytes + (uint32_t)(kk & 3) * 32u) >> 4;
                    mma_bf16_ss(tS, sdesc_make(q_lo + off, kHiK), sdesc_make(k_lo + off, kHiK), idS,
                                kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](uint32_t stage, bool accumulate) {
                const uint32_t v_lo = v_lo0 + stage * (kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk)
                    mma_bf16_ts(tO, tS + (uint32_t)kk * 8u, sdesc_make(v_lo + (uint32_t)kk * (2048u >> 4), kHiV),
                                idPV, (accumulate || kk > 0) ? 1u : 0u);
            };
            const unsigned who = 2u;

            for (long long r = 0; ok; ++r) {
                const long long u = unit_of_round(r, gridDim.x, blockIdx.x);
                if (u >= p.n_units) break;
                const Unit un = w.at(p, r, gridDim.x, blockIdx.x);
                const int n_kv = unit_kv_tiles(p, un);
                if (!wait_poll(bar(kPrepQ ? kBarQReady + t : kBarQFull), unit_it & 1, abort_flag, who, status)) {
                    ok = false;
                    break;
                }
                {
                    const uint32_t s = kv_it % kStages;
                    if (!wait_poll(bar(kBarKvFull + s), (kv_it / kStages) & 1, abort_flag, who, status)) { ok = false; break; }
                    if (!take_turn()) { ok = false; break; }
                    tc_fence_after_sync();
                    issue_s(s);
                    pass_turn();
                    mma_commit(bar(kBarSFull + t));
                    mma_commit(bar(kBarKvEmpty + s));
                    // Q is free once the unit's last Q.K^T completes: the
                    // producer loads the next unit's Q during the last
                    // softmax and P.V instead of after them.
                    if (n_kv == 1) mma_commit(bar(kBarQEmpty));
                }
                for (int j = 0; j < n_kv; ++j) {
                    const uint32_t itv = kv_it + 2u * j + 1u;
                    const uint32_t sv = itv % kStages;
                    const bool more = j + 1 < n_kv;
                    const uint32_t itk = itv + 1u;
                    const uint32_t sk = itk % kStages;
                    if (!wait_poll(bar(kBarKvFull + sv), (itv / kStages) & 1, abort_flag, who, status)) { ok = false; break; }
                    if (more && !wait_poll(bar(kBarKvFull + sk), (itk / kStages) & 1, abort_flag, who, status)) { ok = false; break; }
                    if (!wait_poll(bar(kBarPFull + t), p_phase & 1, abort_flag, who, status)) { ok = false; break; }
                    ++p_phase;
                    if (!take_turn()) { ok = false; break; }
                    tc_fence_after_sync();
                    issue_pv(sv, j > 0);
                    if (more) issue_s(sk);
                    pass_turn();
                    mma_commit(bar(more ? kBarSFull + t : kBarOFull + t));
                    mma_commit(bar(kBarKvEmpty + sv));
                    if (more) mma_commit(bar(kBarKvEmpty + sk));
                    if (j + 2 == n_kv) mma_commit(bar(kBarQEmpty));
                }
                if (!ok) break;
                kv_it += 2u * (uint32_t)n_kv;
                ++unit_it;
            }
            // Nothing this lane issued may still be running when TMEM is freed.
            mma_commit(bar(kBarDrain + t));
            wait_drain(bar(kBarDrain + t), 0, status);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- softmax
        const int t = warp >> 2;                 // query tile of this warpgroup
        const int row = threadIdx.x - 128 * t;   // MMA row = TMEM lane
        const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_bits + (uint32_t)t * 128u;
        const uint32_t tO = tmem + lane_bits + 256u + (uint32_t)t * 128u;
        const int head_in_group = row / p.tile_tokens;
        const int tok_in_tile = row - head_in_group * p.tile_tokens;
        const bool row_used = row < p.tile_rows;
        const float c = p.scale_log2;
        // Q prologue for this thread's row of query tile t of unit `uq`: wait
        // for the tile, RMS-normalise the row and/or rotate it in place in
        // shared memory, then hand the tile to the MMA issuer (the writes go
        // through the generic proxy, the MMA reads through the async proxy).
        auto prep_q = [&](const Unit &uq, uint32_t q_it) -> bool {
            if (!wait_warp(bar(kBarQFull), q_it & 1, abort_flag, 4u, status)) return false;
            const long long tokg = (long long)uq.seq_start + uq.block * p.unit_tokens +
                                   t * p.tile_tokens + tok_in_tile;
            if (row_used && tokg < p.total_tokens) {
                uint8_t *rowp = smem + kQOff + (uint32_t)t * kTileBytes + (uint32_t)row * 128u;
                // 16-byte chunk cc (8 values) of half h of this row, in the
                // 128-byte swizzled layout TMA wrote
                auto chunk = [&](int h, int cc) -> uint4 * {
                    return reinterpret_cast<uint4 *>(rowp + (uint32_t)h * kSubTileBytes +
                                                     (uint32_t)((cc ^ (row & 7)) << 4));
                };
                auto unpack = [](const uint4 v, float (&f)[8]) {
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        f[2 * e] = __uint_as_float(wv[e] << 16);
                        f[2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
                    }
                };
                // the row is read from shared memory once (all 16 chunks in
                // flight), normalised and rotated from registers
                uint4 qa[8], qb[8];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    qa[cc] = *chunk(0, cc);
                    qb[cc] = *chunk(1, cc);
                }
                float rs = 1.0f;
                if (p.q_norm_w != nullptr) {
                    float ss = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        float f[8], g[8];
                        unpack(qa[cc], f);
                        unpack(qb[cc], g);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(g[e], g[e], fmaf(f[e], f[e], ss));
                    }
                    rs = rsqrtf(ss * (1.0f / kHeadDim) + p.norm_eps);
                }
                // element i of the first half pairs with element i + 64 for the
                // rotation, so chunk cc of both halves is processed together
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    float a[8], b[8];
                    unpack(qa[cc], a);
                    unpack(qb[cc], b);
                    if (p.q_norm_w != nullptr) {
                        const uint4 wa = reinterpret_cast<const uint4 *>(smem + kQNormWOff)[cc];
                        const uint4 wb = reinterpret_cast<const uint4 *>(smem + kQNormWOff)[8 + cc];
                        float fa[8], fb[8];
                        unpack(wa, fa);
                        unpack(wb, fb);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            a[e] = a[e] * rs * fa[e];
                            b[e] = b[e] * rs * fb[e];
                        }
                    }
                    if (p.rope_cos != nullptr) {
                        float4 c0, c1, s0, s1;
                        if (p.stage_rope) {
                            // floats 8cc..8cc+7: half cc/4, 16-byte chunks 2(cc%4) and 2(cc%4)+1
                            // of row ur, in the swizzled layout TMA wrote
                            const uint32_t ur = (uint32_t)(t * p.tile_tokens + tok_in_tile);
                            const uint32_t rb = kRopeOff + (uint32_t)(cc >> 2) * kRopeHalfBytes + ur * 128u;
                            const uint32_t k0 = (uint32_t)((2 * (cc & 3)) ^ (ur & 7)) << 4;
                            const uint32_t k1 = (uint32_t)((2 * (cc & 3) + 1) ^ (ur & 7)) << 4;
                            c0 = *reinterpret_cast<const float4 *>(smem + rb + k0);
                            c1 = *reinterpret_cast<const float4 *>(smem + rb + k1);
                            s0 = *reinterpret_cast<const float4 *>(smem + rb + 2 * kRopeHalfBytes + k0);
                            s1 = *reinterpret_cast<const float4 *>(smem + rb + 2 * kRopeHalfBytes + k1);
                        } else {
                            const float4 *cs4 = reinterpret_cast<const float4 *>(p.rope_cos + tokg * (kHeadDim / 2) + 8 * cc);
                            const float4 *sn4 = reinterpret_cast<const float4 *>(p.rope_sin + tokg * (kHeadDim / 2) + 8 * cc);
                            c0 = __ldg(cs4); c1 = __ldg(cs4 + 1); s0 = __ldg(sn4); s1 = __ldg(sn4 + 1);
                        }
                        const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float x0 = a[e], x1 = b[e];
                            a[e] = x0 * cs[e] - x1 * sn[e];
                            b[e] = x1 * cs[e] + x0 * sn[e];
                        }
                    }
                    *chunk(0, cc) = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                               pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
                    *chunk(1, cc) = make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]),
                                               pack_bf16x2(b[4], b[5]), pack_bf16x2(b[6], b[7]));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarQReady + t));
            return true;
        };

        // The schedule state lives in this thread's shared-memory slot: it is
        // used once per unit, and the registers are needed by the score rows.
        Schedule &w = reinterpret_cast<Schedule *>(smem + kSchedOff)[threadIdx.x];
        w.init(p);
        uint32_t s_phase = 0, o_phase = 0, q_it = 0;
        bool ok = true;
        // Each unit is looked up at the end of the one before, where the
        // score rows are no longer live.
        Unit un;
        const int grid = gridDim.x, cta = blockIdx.x;
        if (unit_of_round(0, grid, cta) < p.n_units) {
            un = w.at(p, 0, grid, cta);
            if (kPrepQ) ok = prep_q(un, 0);
        }
        for (long long r = 0; ok; ++r) {
            if (unit_of_round(r, grid, cta) >= p.n_units) break;
            const int tb = un.block * p.unit_tokens;
            const int n_kv = unit_kv_tiles(p, un);
            const int tok = tb + t * p.tile_tokens + tok_in_tile;   // token inside its sequence
            // key tiles from here on may hold keys a row must not see: past
            // the unit's first token (causal; one tile when the unit size
            // divides 128, at most two otherwise) or past the sequence end
            const int mask_from = p.causal ? (tb >> 7) : n_kv - 1;
            float m = -INFINITY;   // running max of the scaled logits, log2 units
            float l = 0.f;         // running sum of exp2(logit - m)
            for (int j = 0; j < n_kv; ++j) {
                if (!wait_warp(bar(kBarSFull + t), s_phase & 1, abort_flag, 4u, status)) { ok = false; break; }
                ++s_phase;
                tc_fence_after_sync();
                float s[kKeys];
                {
                    uint32_t sr[kKeys];
                    tmem_ld128_wait(tS, sr);
#pragma unroll
                    for (int i = 0; i < kKeys; ++i) s[i] = __uint_as_float(sr[i]);
                }
                if (j >= mask_from) {
                    // key (j*128 + i) is visible iff it is <= tok (causal) or
                    // inside the sequence (bidirectional)
                    const int lim = (p.causal ? tok : un.seq_len - 1) - j * kKeys;
#pragma unroll
                    for (int i = 0; i < kKeys; ++i)
                        if (i > lim) s[i] = -INFINITY;
                }
                // row max: four running maxima over s[a + 4k], k = 0..31
                float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int k = 1; k + 1 < kKeys / 4; k += 2) {
#pragma unroll
                    for (int a = 0; a < 4; ++a) mx[a] = max3(mx[a], s[4 * k + a], s[4 * k + 4 + a]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) mx[a] = fmaxf(mx[a], s[kKeys - 4 + a]);
                const float m_tile = max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * c;
                const float m_new = fmaxf(m, m_tile);
                float m_use = m, alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_use = m_new;
                } else if (m_new - m > kRescaleThreshold) {
                    m_use = m_new;
                    alpha = ex2_approx(m - m_new);
                    rescale = true;
                }
                // p = 2^(s*c - m_use), two lanes at a time on the packed FMA
                // path; the fp32 p feed the row sum, their bf16 rounding is P.
                const float2 c2 = make_float2(c, c);
                const float2 nm2 = make_float2(-m_use, -m_use);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
                uint32_t pk[kKeys / 2];
#pragma unroll
                for (int i = 0; i < kKeys / 2; ++i) {
                    const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), c2, nm2);
                    const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    if (i & 1) acc1 = __fadd2_rn(acc1, e); else acc0 = __fadd2_rn(acc0, e);
                    pk[i] = pack_bf16x2(e.x, e.y);
                    if ((i & 15) == 15) tmem_st16(tS + (uint32_t)(i - 15), &pk[i - 15]);
                }
                const float2 acc = __fadd2_rn(acc0, acc1);
                l = l * alpha + (acc.x + acc.y);
                m = m_use;
                if (__any_sync(0xffffffffu, rescale)) {
                    // PV of the previous tile is complete (it was issued
                    // before this S), so O can be scaled in place.
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t rr[32];
                        tmem_ld32_wait(tO + (uint32_t)ch * 32u, rr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
                        tmem_st32(tO + (uint32_t)ch * 32u, rr);
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(bar(kBarPFull + t));
            }
            if (!ok) break;
            // The next unit's Q tile lands while this unit's last P.V and the
            // epilogue run; its rotary table rows are pulled into L1 now.
            ++q_it;
            const bool has_next = unit_of_round(r + 1, grid, cta) < p.n_units;
            const bool prep_next = kPrepQ && has_next;
            Unit next_un = un;
            if (prep_next) {
                next_un = w.at(p, r + 1, grid, cta);
                if (p.rope_cos != nullptr && !p.stage_rope) {
                    const long long tn = (long long)next_un.seq_start + next_un.block * p.unit_tokens +
                                         t * p.tile_tokens + tok_in_tile;
                    if (tn < p.total_tokens) {
#pragma unroll
                        for (int li = 0; li < 2; ++li) {
                            prefetch_l1(p.rope_cos + tn * (kHeadDim / 2) + li * 32);
                            prefetch_l1(p.rope_sin + tn * (kHeadDim / 2) + li * 32);
                        }
                    }
                }
            }
            // ------------------------------------------------------ epilogue
            if (!wait_warp(bar(kBarOFull + t), o_phase & 1, abort_flag, 4u, status)) { ok = false; break; }
            ++o_phase;
            tc_fence_after_sync();
            const float inv_l = 1.0f / l;
            const bool valid = row_used && tok < un.seq_len;
            const int head = (p.group0 + un.group) * p.tile_heads + head_in_group;
            const long long tok_g = (long long)un.seq_start + tok;
            const long long grow = (long long)head * p.total_tokens + tok_g;          // [Hq][T] index
            const long long orow = p.out_token_major ? tok_g * p.n_q_heads + head : grow;
            if (!kInt8) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) + orow * kHeadDim);
                // a rolled loop: this code runs once per unit, and less of it
                // is fetched at the unit boundary (paired: +0.1 to +0.9%)
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t rr[32];
                    tmem_ld32_wait(tO + (uint32_t)ch * 32u, rr);
                    if (valid) {
                        uint4 pk4[4];
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 pkt;
                            pkt.x = pack_bf16x2(__uint_as_float(rr[v4 * 8 + 0]) * inv_l, __uint_as_float(rr[v4 * 8 + 1]) * inv_l);
                            pkt.y = pack_bf16x2(__uint_as_float(rr[v4 * 8 + 2]) * inv_l, __uint_as_float(rr[v4 * 8 + 3]) * inv_l);
                            pkt.z = pack_bf16x2(__uint_as_float(rr[v4 * 8 + 4]) * inv_l, __uint_as_float(rr[v4 * 8 + 5]) * inv_l);
                            pkt.w = pack_bf16x2(__uint_as_float(rr[v4 * 8 + 6]) * inv_l, __uint_as_float(rr[v4 * 8 + 7]) * inv_l);
                            pk4[v4] = pkt;
                        }
                        // 32-byte stores (whole L2 sectors) when o allows it
                        if (p.o_align32 && !kPrepQ) {
                            // O is written once and not read here again: first
                            // out of L2
                            const uint64_t pol_o = l2_policy_evict_first();
                            stg256_hint(dst + ch * 4, pk4[0], pk4[1], pol_o);
                            stg256_hint(dst + ch * 4 + 2, pk4[2], pk4[3], pol_o);
                        } else if (p.o_align32) {
                            stg256(dst + ch * 4, pk4[0], pk4[1]);
                            stg256(dst + ch * 4 + 2, pk4[2], pk4[3]);
                        } else {
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) dst[ch * 4 + v4] = pk4[v4];
                        }
                    }
                }
            } else {
                // int8 with one scale per (token, head) row: scale = max|o| / 127,
                // code = round-to-nearest-even(o / scale), o ~= code * scale.
                float x[kHeadDim];
                {
                    uint32_t rr[kHeadDim];
                    tmem_ld128_wait(tO, rr);
#pragma unroll
                    for (int i = 0; i < kHeadDim; ++i) x[i] = __uint_as_float(rr[i]) * inv_l;
                }
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < kHeadDim; ++i) amax = fmaxf(amax, fabsf(x[i]));
                const float qscale = amax > 0.f ? amax / 127.0f : 1.0f;
                // 127 / max|o| is finite for max|o| > 3.75e-37; a row below
                // that gets all-zero codes (within 3.75e-37 of o)
                const float inv_q = amax > 3.75e-37f ? 127.0f / amax : 0.0f;
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<int8_t *>(p.o) + orow * kHeadDim);
                    // t = x * inv_q lies in [-127, 127] up to the product's
                    // rounding (it cannot reach 127.5), so adding 1.5 * 2^23
                    // rounds it to the nearest integer, ties to even, and
                    // leaves that integer's two's-complement low byte in the
                    // low byte of the sum's bits: the same code as converting
                    // t to an integer, on the FMA pipe instead of the
                    // conversion unit. Separate multiply and add (never
                    // contracted) keep t rounded to fp32 first.
                    constexpr float kRound = 12582912.0f;
#pragma unroll
                    for (int v4 = 0; v4 < kHeadDim / 16; ++v4) {
                        uint32_t w4[4];
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            uint32_t b[4];
#pragma unroll
                            for (int bi = 0; bi < 4; ++bi)
                                b[bi] = __float_as_uint(__fadd_rn(__fmul_rn(x[v4 * 16 + wi * 4 + bi], inv_q), kRound));
                            w4[wi] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
                        }
                        dst[v4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    p.o_scale[orow] = qscale;
                }
            }
            if (valid) p.lse[grow] = (m + __log2f(l)) * 0.69314718055994531f;
            tc_fence_before_sync();
            if (prep_next && !prep_q(next_un, q_it)) { ok = false; break; }
            if (has_next && !prep_next) next_un = w.at(p, r + 1, grid, cta);
            un = next_un;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace h3gqa
