// Host side of the h3gqa C ABI: argument checks, the work plan, TMA tensor
// maps and the launch of the sm_103a causal GQA kernel.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/h3gqa.h"
#include "fwd_kernel.cuh"
#include "prep_kernel.cuh"

namespace {

using h3gqa::FwdParams;

constexpr int kVersion = 10100;   // 1.1.0
constexpr long long kMaxTotalTokens = (1LL << 31) - 256;
constexpr long long kMaxUnits = (1LL << 31) - 1;

struct HostPlan {
    int group = 0;             // G = Hq / Hkv
    int tile_heads = 0;        // query heads per tile: the largest divisor of G that is <= 128
    int tile_tokens = 0;       // floor(128 / tile_heads)
    int unit_tokens = 0;       // 2 * tile_tokens
    bool pow2 = false;         // unit_tokens is a power of two that divides 128
    int blocks_per_class = 0;  // pow2 only
    int c_max = 0;             // cost class of the longest sequence's last block
    int max_kv_tiles = 0;      // most key tiles any unit visits
    int n_groups = 0;          // head groups of the call (all KV heads, or the shard's)
    long long n_units = 0;
    long long n_kv_tiles = 0;
    long long total_tokens = 0;
    std::vector<int> start;   // non-empty sequences, longest first
    std::vector<int> len;
};

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int x)
{
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

int largest_divisor_upto(int g, int cap)
{
    for (int d = std::min(g, cap); d > 1; --d)
        if (g % d == 0) return d;
    return 1;
}

// Shape checks shared by the plan query and the forward call; no CUDA.
// kv_count KV heads (from any first head) are planned; the caller checks the
// range against n_kv_heads.
h3gqa_status build_plan(const int32_t *cu, int n_seqs, int hq, int hkv, int head_dim,
                        bool causal, int kv_count, HostPlan *out)
{
    if (cu == nullptr || n_seqs < 0) return H3GQA_ERR_INVALID_ARG;
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return H3GQA_ERR_INVALID_ARG;
    if (head_dim <= 0) return H3GQA_ERR_INVALID_ARG;
    if (cu[0] != 0) return H3GQA_ERR_INVALID_ARG;
    for (int b = 0; b < n_seqs; ++b)
        if (cu[b + 1] < cu[b]) return H3GQA_ERR_INVALID_ARG;
    if (head_dim != h3gqa::kHeadDim) return H3GQA_ERR_UNSUPPORTED;
    const long long T = cu[n_seqs];
    if (T > kMaxTotalTokens) return H3GQA_ERR_UNSUPPORTED;

    HostPlan p;
    p.group = hq / hkv;
    p.tile_heads = largest_divisor_upto(p.group, h3gqa::kRows);
    p.tile_tokens = h3gqa::kRows / p.tile_heads;
    p.unit_tokens = 2 * p.tile_tokens;
    p.pow2 = is_pow2(p.unit_tokens) && p.unit_tokens <= h3gqa::kKeys;
    p.blocks_per_class = p.pow2 ? h3gqa::kKeys / p.unit_tokens : 0;
    p.n_groups = kv_count * (p.group / p.tile_heads);
    p.total_tokens = T;
    std::vector<int> order;
    for (int b = 0; b < n_seqs; ++b)
        if (cu[b + 1] > cu[b]) order.push_back(b);
    if ((int)order.size() > h3gqa::kMaxSeqs) return H3GQA_ERR_UNSUPPORTED;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        return (cu[a + 1] - cu[a]) > (cu[b + 1] - cu[b]);
    });
    const long long U = p.unit_tokens;
    for (int b : order) {
        const int len = cu[b + 1] - cu[b];
        p.start.push_back(cu[b]);
        p.len.push_back(len);
        const long long nblk = (len + U - 1) / U;
        p.n_units += nblk * p.n_groups;
        if (causal) {
            // block k visits the key tiles up to its last token in the sequence
            for (long long k = 0; k < nblk; ++k) {
                const long long tiles = std::min(k * U + U, (long long)len) - 1;
                p.n_kv_tiles += (tiles / h3gqa::kKeys + 1) * p.n_groups;
                p.max_kv_tiles = std::max(p.max_kv_tiles, (int)(tiles / h3gqa::kKeys + 1));
            }
        } else {
            const long long tiles = (len + h3gqa::kKeys - 1) / h3gqa::kKeys;
            p.n_kv_tiles += nblk * tiles * p.n_groups;
            p.max_kv_tiles = std::max(p.max_kv_tiles, (int)tiles);
        }
    }
    // the kernel counts units and rounds in 32-bit integers
    if (p.n_units > kMaxUnits) return H3GQA_ERR_UNSUPPORTED;
    if (!p.len.empty()) {
        const long long nblk0 = (p.len[0] + U - 1) / U;
        p.c_max = causal ? (int)((nblk0 * U - 1) / h3gqa::kKeys + 1)
                         : (p.len[0] + h3gqa::kKeys - 1) / h3gqa::kKeys;
    }
    *out = std::move(p);
    return H3GQA_OK;
}

// ------------------------------------------------------------ per device
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    h3gqa_status status = H3GQA_OK;
    int sm_count = 0;
};

// A fixed table, so a DeviceState handed out stays where it is while other
// threads set up other devices.
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

h3gqa_status device_setup(int dev, DeviceState **out, bool again = false)
{
    if (dev < 0 || dev >= kMaxDevices) return H3GQA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (again && d.ready && d.status == H3GQA_OK) d.ready = false;
    if (d.ready) {
        *out = &d;
        return d.status;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return H3GQA_ERR_CUDA;
    d.ready = true;
    d.sm_count = sms;
    if (major != 10 || minor != 3) {
        d.status = H3GQA_ERR_ARCH;
        *out = &d;
        return d.status;
    }
    if (cudaFuncSetAttribute(h3gqa::causal_gqa_fwd_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h3gqa::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(h3gqa::causal_gqa_fwd_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h3gqa::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(h3gqa::causal_gqa_fwd_kernel<true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h3gqa::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(h3gqa::causal_gqa_fwd_kernel<true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h3gqa::kSmemBytes) != cudaSuccess) {
        d.ready = false;
        return H3GQA_ERR_CUDA;
    }
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
            d.ready = false;
            return H3GQA_ERR_CUDA;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.status = H3GQA_OK;
    *out = &d;
    return H3GQA_OK;
}

// A [heads][T][128] bf16 tensor as a 3-D TMA map with a {64, rows, heads}
// box and the 128-byte swizzle that the tcgen05 descriptors expect.
bool encode_map(CUtensorMap *map, const void *base, int heads, long long T,
                int box_rows, int box_heads)
{
    cuuint64_t dims[3] = {(cuuint64_t)h3gqa::kHeadDim, (cuuint64_t)T, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)h3gqa::kHeadDim * 2,
                             (cuuint64_t)T * h3gqa::kHeadDim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_heads};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tiling and unit-schedule fields of the kernel parameters for a plan
// (no CUDA): KV heads from kv_begin, a persistent grid of at most sm_count
// CTAs. Returns the grid size (n_units > 0).
int fill_schedule(const HostPlan &hp, int kv_begin, int sm_count, FwdParams *prm)
{
    prm->total_tokens = hp.total_tokens;
    prm->n_units = hp.n_units;
    prm->n_groups = hp.n_groups;
    prm->groups_per_kv = hp.group / hp.tile_heads;
    prm->group0 = kv_begin * prm->groups_per_kv;
    prm->tile_heads = hp.tile_heads;
    prm->tile_tokens = hp.tile_tokens;
    prm->tile_rows = hp.tile_heads * hp.tile_tokens;
    prm->unit_tokens = hp.unit_tokens;
    prm->pow2 = hp.pow2 ? 1 : 0;
    prm->unit_tokens_log2 = hp.pow2 ? ilog2(hp.unit_tokens) : 0;
    prm->blocks_per_class = hp.blocks_per_class;
    prm->blocks_per_class_log2 = hp.pow2 ? ilog2(hp.blocks_per_class) : 0;
    prm->q_tx_bytes = 2u * 2u * (unsigned)prm->tile_rows * 128u;   // 2 tiles x 2 halves x rows x 128 B
    prm->n_seqs = (int)hp.len.size();
    prm->c_max = hp.c_max;
    for (size_t i = 0; i < hp.len.size(); ++i) {
        prm->seq_start[i] = hp.start[i];
        prm->seq_len[i] = hp.len[i];
    }
    const int grid = (int)std::min<long long>(hp.n_units, sm_count);
    prm->full_windows = (int)(hp.n_units / hp.n_groups / grid);
    return grid;
}

// A rotary table fp32 [T][64] as a 2-D map with {32, 32} boxes (32 rows of
// one 128-byte half) and the 128-byte swizzle the Q prologue reads.
bool encode_map_rope(CUtensorMap *map, const float *base, long long T)
{
    cuuint64_t dims[2] = {(cuuint64_t)h3gqa::kHeadDim / 2, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)h3gqa::kHeadDim / 2 * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)h3gqa::kRopeMaxTokens};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a + na) and [b, b + nb) share a byte
bool overlaps(const void *a, unsigned long long na, const void *b, unsigned long long nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

h3gqa_status h3gqa_attention_plan(const int32_t *cu_seqlens, int n_seqs, int n_q_heads,
                                  int n_kv_heads, int head_dim, int32_t causal, h3gqa_plan *plan)
{
    if (plan == nullptr || (causal != 0 && causal != 1)) return H3GQA_ERR_INVALID_ARG;
    HostPlan hp;
    const h3gqa_status st = build_plan(cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim,
                                       causal != 0, n_kv_heads, &hp);
    if (st != H3GQA_OK) return st;
    std::memset(plan, 0, sizeof(*plan));
    plan->total_tokens = hp.total_tokens;
    plan->n_units = hp.n_units;
    plan->n_kv_tiles = hp.n_kv_tiles;
    plan->tensor_flops = (double)hp.n_kv_tiles * 2.0 * 2.0 * 2.0 * 128.0 * 128.0 * 128.0;
    double needed = 0, metric = 0, ex = 0;
    for (int len : hp.len) {
        const double S = (double)len;
        if (causal) {
            needed += 2.0 * n_q_heads * head_dim * S * (S + 1.0);
            metric += 2.0 * n_q_heads * head_dim * S * S;
            ex += (double)n_q_heads * S * (S + 1.0) / 2.0;
        } else {
            needed += 4.0 * n_q_heads * head_dim * S * S;
            metric += 4.0 * n_q_heads * head_dim * S * S;
            ex += (double)n_q_heads * S * S;
        }
    }
    plan->causal_flops = needed;
    plan->metric_flops = metric;
    plan->exp2_count = ex;
    const double T = (double)hp.total_tokens;
    plan->algorithmic_bytes = 2.0 * T * head_dim * (2.0 * n_q_heads + 2.0 * n_kv_heads) +
                              4.0 * T * n_q_heads;
    plan->tokens_per_unit = hp.unit_tokens;
    plan->max_kv_tiles = hp.max_kv_tiles;
    plan->heads_per_tile = hp.tile_heads;
    plan->rows_per_tile = hp.tile_heads * hp.tile_tokens;
    return H3GQA_OK;
}

h3gqa_status h3gqa_make_plan(const int32_t *cu_seqlens, int n_seqs, int n_q_heads,
                             int n_kv_heads, int head_dim, h3gqa_plan *plan)
{
    return h3gqa_attention_plan(cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim, 1, plan);
}

h3gqa_status h3gqa_attention_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                                 const int32_t *cu_seqlens, int n_seqs, int n_q_heads,
                                 int n_kv_heads, int head_dim, float scale,
                                 const h3gqa_options *options, h3gqa_stream_t stream)
{
    h3gqa_options opt;
    std::memset(&opt, 0, sizeof(opt));
    opt.causal = 1;
    opt.out_layout = H3GQA_LAYOUT_HEAD_MAJOR;
    if (options != nullptr) opt = *options;
    const bool prep_k = opt.k_norm_weight != nullptr || opt.rope_cos != nullptr;
    const bool prep_q = opt.q_norm_weight != nullptr || opt.rope_cos != nullptr;
    if ((opt.rope_cos == nullptr) != (opt.rope_sin == nullptr) ||
        !aligned(opt.q_norm_weight, 16) || !aligned(opt.k_norm_weight, 16) ||
        !aligned(opt.rope_cos, 16) || !aligned(opt.rope_sin, 16) ||
        (prep_k && (opt.k_out == nullptr || !aligned(opt.k_out, 16))) ||
        !(opt.norm_eps >= 0.0f) || !std::isfinite(opt.norm_eps))
        return H3GQA_ERR_INVALID_ARG;
    if ((opt.causal != 0 && opt.causal != 1) || !aligned(opt.status, 4) ||
        (opt.out_layout != H3GQA_LAYOUT_HEAD_MAJOR && opt.out_layout != H3GQA_LAYOUT_TOKEN_MAJOR) ||
        (opt.out_int8 != 0 && opt.out_int8 != 1))
        return H3GQA_ERR_INVALID_ARG;
    if (opt.out_int8 && (opt.o_scale == nullptr || !aligned(opt.o_scale, 4)))
        return H3GQA_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !lse) return H3GQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(lse, 4))
        return H3GQA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return H3GQA_ERR_INVALID_ARG;
    // head shard: KV heads [kv_begin, kv_begin + kv_count)
    if (n_kv_heads <= 0 || opt.kv_head_begin < 0 || opt.kv_head_count < 0 ||
        opt.kv_head_begin >= n_kv_heads ||
        opt.kv_head_count > n_kv_heads - opt.kv_head_begin)
        return H3GQA_ERR_INVALID_ARG;
    const int kv_begin = opt.kv_head_begin;
    const int kv_count = opt.kv_head_count ? opt.kv_head_count : n_kv_heads - kv_begin;
    HostPlan hp;
    h3gqa_status st = build_plan(cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim,
                                 opt.causal != 0, kv_count, &hp);
    if (st != H3GQA_OK) return st;
    {
        // prepared keys go to their own buffer or over k itself, never over
        // q, v or part of k
        const unsigned long long T = (unsigned long long)hp.total_tokens;
        const unsigned long long qb = 2ull * n_q_heads * T * head_dim;
        const unsigned long long kb = 2ull * n_kv_heads * T * head_dim;
        if (prep_k && T > 0 &&
            (overlaps(opt.k_out, kb, q, qb) || overlaps(opt.k_out, kb, v, kb) ||
             (opt.k_out != k && overlaps(opt.k_out, kb, k, kb))))
            return H3GQA_ERR_INVALID_ARG;
        // o is written while other units still read q, k and v
        const unsigned long long ob = (opt.out_int8 ? 1ull : 2ull) * n_q_heads * T * head_dim;
        const unsigned long long lb = 4ull * n_q_heads * T;
        if (T > 0 && (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kb) || overlaps(o, ob, v, kb) ||
                      overlaps(o, ob, lse, lb) || (prep_k && overlaps(o, ob, opt.k_out, kb)) ||
                      (opt.out_int8 && overlaps(o, ob, opt.o_scale, lb))))
            return H3GQA_ERR_INVALID_ARG;
    }
    if (hp.n_units == 0) return H3GQA_OK;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return H3GQA_ERR_CUDA;
    DeviceState *ds = nullptr;
    st = device_setup(dev, &ds);
    if (st != H3GQA_OK) return st;

    const long long T = hp.total_tokens;
    const void *k_used = k;
    if (prep_k) {
        // keys once, into k_out, before the attention reads them (the
        // shard's KV heads only)
        const long long rows = (long long)kv_count * T;
        const long long first = (long long)kv_begin * T * head_dim;
        // one row per warp: every row's loads are in flight at once
        const long long blocks = std::min<long long>((rows + 7) / 8, 1LL << 30);
        h3gqa::qk_prep_kernel<<<(unsigned)blocks, h3gqa::kPrepThreads, 0,
                                reinterpret_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint16_t *>(k) + first, static_cast<uint16_t *>(opt.k_out) + first, rows, T,
            static_cast<const uint16_t *>(opt.k_norm_weight), opt.norm_eps, opt.rope_cos,
            opt.rope_sin);
        if (cudaGetLastError() != cudaSuccess) return H3GQA_ERR_CUDA;
        k_used = opt.k_out;
    }
    FwdParams *prm = new (std::nothrow) FwdParams;
    if (prm == nullptr) return H3GQA_ERR_CUDA;
    std::memset(prm, 0, sizeof(*prm));
    if (!encode_map(&prm->map_q, q, n_q_heads, T, hp.tile_tokens, hp.tile_heads) ||
        !encode_map(&prm->map_k, k_used, n_kv_heads, T, h3gqa::kKeys, 1) ||
        !encode_map(&prm->map_v, v, n_kv_heads, T, h3gqa::kKeys, 1)) {
        delete prm;
        return H3GQA_ERR_CUDA;
    }
    prm->o = o;
    prm->lse = lse;
    prm->o_scale = opt.o_scale;
    prm->status = opt.status;
    prm->causal = opt.causal;
    prm->out_token_major = opt.out_layout == H3GQA_LAYOUT_TOKEN_MAJOR;
    prm->out_int8 = opt.out_int8;
    prm->o_align32 = aligned(o, 32) ? 1 : 0;
    prm->n_q_heads = n_q_heads;
    prm->prep_q = prep_q ? 1 : 0;
    prm->stage_rope = (opt.rope_cos != nullptr && hp.unit_tokens <= h3gqa::kRopeMaxTokens) ? 1 : 0;
    if (prm->stage_rope && (!encode_map_rope(&prm->map_cos, opt.rope_cos, T) ||
                            !encode_map_rope(&prm->map_sin, opt.rope_sin, T))) {
        delete prm;
        return H3GQA_ERR_CUDA;
    }
    prm->q_norm_w = static_cast<const uint16_t *>(opt.q_norm_weight);
    prm->rope_cos = opt.rope_cos;
    prm->rope_sin = opt.rope_sin;
    prm->norm_eps = opt.norm_eps;
    prm->scale_log2 = scale * 1.4426950408889634f;
    const int grid = fill_schedule(hp, kv_begin, ds->sm_count, prm);
    // the instance for this call's output dtype and Q prologue
    void (*kernel)(const FwdParams) =
        prm->out_int8 ? (prm->prep_q ? h3gqa::causal_gqa_fwd_kernel<true, true>
                                     : h3gqa::causal_gqa_fwd_kernel<true, false>)
                      : (prm->prep_q ? h3gqa::causal_gqa_fwd_kernel<false, true>
                                     : h3gqa::causal_gqa_fwd_kernel<false, false>);
    kernel<<<(unsigned)grid, h3gqa::kThreads, h3gqa::kSmemBytes,
             reinterpret_cast<cudaStream_t>(stream)>>>(*prm);
    cudaError_t err = cudaGetLastError();
    if (err == cudaErrorInvalidValue || err == cudaErrorLaunchOutOfResources) {
        // The kernel's shared-memory attribute is per context: after a device
        // reset it is gone although this table still says ready. Set the
        // device up again and launch once more.
        if (device_setup(dev, &ds, true) == H3GQA_OK) {
            kernel<<<(unsigned)grid, h3gqa::kThreads, h3gqa::kSmemBytes,
                     reinterpret_cast<cudaStream_t>(stream)>>>(*prm);
            err = cudaGetLastError();
        }
    }
    delete prm;
    return err == cudaSuccess ? H3GQA_OK : H3GQA_ERR_CUDA;
}

h3gqa_status h3gqa_causal_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int n_seqs, int n_q_heads,
                              int n_kv_heads, int head_dim, float scale, h3gqa_stream_t stream)
{
    return h3gqa_attention_fwd(q, k, v, o, lse, cu_seqlens, n_seqs, n_q_heads, n_kv_heads,
                               head_dim, scale, nullptr, stream);
}

h3gqa_status h3gqa_sync_and_check(h3gqa_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return H3GQA_ERR_CUDA;
    unsigned int flags = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&flags, h3gqa::g_timeout_flags, sizeof(flags)) != cudaSuccess)
        return H3GQA_ERR_CUDA;
    if (flags != 0 &&
        cudaMemcpyToSymbol(h3gqa::g_timeout_flags, &zero, sizeof(zero)) != cudaSuccess)
        return H3GQA_ERR_CUDA;
    return flags ? H3GQA_ERR_TIMEOUT : H3GQA_OK;
}

const char *h3gqa_status_string(h3gqa_status s)
{
    switch (s) {
    case H3GQA_OK: return "ok";
    case H3GQA_ERR_INVALID_ARG: return "invalid argument";
    case H3GQA_ERR_UNSUPPORTED: return "unsupported shape (head_dim must be 128, at most 1024 non-empty sequences, T < 2^31 - 256)";
    case H3GQA_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case H3GQA_ERR_CUDA: return "CUDA call failed";
    case H3GQA_ERR_TIMEOUT: return "kernel gave up on a bounded internal wait";
    }
    return "unknown status";
}

int h3gqa_version(void) { return kVersion; }

}  // extern "C"
