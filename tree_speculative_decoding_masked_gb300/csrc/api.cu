// C ABI of libtreeverify: host-side argument checks, workspace carving and launches.
// Nothing here allocates device memory, synchronises the stream or throws.
#include <math.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "tv_kernels.cuh"

using namespace tv;

// Process-wide settings, read at every launch (atomics: another host thread may change
// them while launches are being made).
// SM shares for running the vocab pass and the tree attention concurrently (0 = all SMs)
static std::atomic<int> g_sm_verify{0}, g_sm_attention{0};
// tensor-core attention kernel: 0 automatic, 1 one row tile per CTA, 2 paired row tiles,
// 3 paired row tiles with 64-key KV tiles and double-buffered S, 4 variant 3 on a
// persistent grid
static std::atomic<int> g_attn_variant{0};
// KV splits per tensor-core attention CTA group: 0 automatic, else forced (capped at the
// KV tile count and the cluster limit)
static std::atomic<int> g_attn_splits{0};

namespace tv {
int sm_share_verify() { return g_sm_verify.load(std::memory_order_relaxed); }
int sm_share_attention() { return g_sm_attention.load(std::memory_order_relaxed); }
int attention_variant() { return g_attn_variant.load(std::memory_order_relaxed); }
int attention_splits() { return g_attn_splits.load(std::memory_order_relaxed); }
}  // namespace tv

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_dtype(tv_dtype d) { return d == TV_F32 || d == TV_BF16; }
inline tv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TV_OK : TV_ERR_CUDA; }
inline cudaStream_t st(tv_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// One NVTX range per entry point that launches work, named after the entry point, so
// that a profiler's timeline groups each call's kernels.  NVTX is header-only: without an
// attached tool a push or pop is one pointer check.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace

extern "C" {

const char* tv_status_string(int s) {
  switch (s) {
    case TV_OK:
      return "TV_OK";
    case TV_ERR_NULL:
      return "TV_ERR_NULL: a required pointer is NULL";
    case TV_ERR_SHAPE:
      return "TV_ERR_SHAPE: a size is outside the supported range";
    case TV_ERR_DTYPE:
      return "TV_ERR_DTYPE: unsupported dtype";
    case TV_ERR_WORKSPACE:
      return "TV_ERR_WORKSPACE: workspace missing or too small";
    case TV_ERR_ALIGN:
      return "TV_ERR_ALIGN: pointer or stride misaligned";
    case TV_ERR_UNSUPPORTED:
      return "TV_ERR_UNSUPPORTED: combination not implemented";
    case TV_ERR_CUDA:
      return "TV_ERR_CUDA: CUDA call failed while enqueueing";
    case TV_ERR_VALUE:
      return "TV_ERR_VALUE: scalar argument out of range";
    default:
      return "unknown tv_status";
  }
}

int tv_version(void) { return (1 << 16) | 0; }

tv_status tv_philox4x32_10(uint64_t seed, const uint32_t* counters, int n, uint32_t* out, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_philox4x32_10");
  if (n < 0) return TV_ERR_SHAPE;
  if (n > 0 && (!counters || !out)) return TV_ERR_NULL;
  if (!aligned16(counters) || !aligned16(out)) return TV_ERR_ALIGN;
  return cuda_status(launch_philox_words(seed, counters, n, out, st(stream)));
}

tv_status tv_selftest_bounded_wait(int wait_us, int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_selftest_bounded_wait");
  if (!dev_status) return TV_ERR_NULL;
  if (wait_us < 1 || wait_us > 1000000) return TV_ERR_VALUE;
  return cuda_status(launch_wait_selftest((uint64_t)wait_us * 1000ull, dev_status, st(stream)));
}

tv_status tv_set_sm_partition(int verify_sms, int attention_sms) {
  if (verify_sms < 0 || attention_sms < 0) return TV_ERR_VALUE;
  g_sm_verify.store(verify_sms, std::memory_order_relaxed);
  g_sm_attention.store(attention_sms, std::memory_order_relaxed);
  return TV_OK;
}

tv_status tv_set_attention_variant(int variant) {
  if (variant < 0 || variant > 5) return TV_ERR_VALUE;
  g_attn_variant.store(variant, std::memory_order_relaxed);
  return TV_OK;
}

tv_status tv_set_attention_splits(int splits) {
  if (splits < 0 || splits > 8) return TV_ERR_VALUE;
  g_attn_splits.store(splits, std::memory_order_relaxed);
  return TV_OK;
}

tv_status tv_tree_prep(const int32_t* parent, int B, int N, int P, int32_t* depth, int32_t* pos, uint32_t* anc_mask,
                       int32_t* child_off, int32_t* child_idx, int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_tree_prep");
  if (!parent) return TV_ERR_NULL;
  if (B < 1 || N < 1 || N > kMaxNodes || P < 0) return TV_ERR_SHAPE;
  if ((child_off == nullptr) != (child_idx == nullptr)) return TV_ERR_NULL;
  return cuda_status(launch_tree_prep(parent, B, N, P, depth, pos, anc_mask, child_off, child_idx, dev_status,
                                      st(stream)));
}

tv_status tv_prune_tree(const int32_t* parent, const float* conf, int B, int N, int max_children, int depth_limit,
                        int32_t* old_to_new, int32_t* new_parent, int32_t* n_kept, int32_t* new_root,
                        int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_prune_tree");
  if (!parent || !conf || !old_to_new || !new_parent || !n_kept || !new_root) return TV_ERR_NULL;
  if (B < 1 || N < 1 || N > kMaxNodes) return TV_ERR_SHAPE;
  if (max_children < 1 || depth_limit < 1) return TV_ERR_VALUE;
  return cuda_status(launch_prune(parent, conf, B, N, max_children, depth_limit, old_to_new, new_parent, n_kept,
                                  new_root, dev_status, st(stream)));
}

size_t tv_tree_attention_workspace_size(int B, int Hq, int Hkv, int D, int P, int N, tv_dtype dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || P < 0 || N < 1) return 0;
  AttnPlan p = attn_plan(B, Hq, Hkv, D, P, N, dtype);
  return p.tc ? p.total : 0;
}

tv_status tv_tree_attention(const void* q, const void* k_cache, const void* v_cache, void* out,
                            const int32_t* parent, int B, int Hq, int Hkv, int D, int P, int N, int kv_stride_tokens,
                            float scale, tv_dtype dtype, void* workspace, size_t ws_bytes, int32_t* dev_status,
                            tv_stream_t stream) {
  NvtxRange nvtx_range("tv_tree_attention");
  if (!q || !k_cache || !v_cache || !out || !parent) return TV_ERR_NULL;
  if (!valid_dtype(dtype)) return TV_ERR_DTYPE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || N < 1 || N > kMaxNodes || P < 0) return TV_ERR_SHAPE;
  if (D < 32 || D > 256 || D % 32) return TV_ERR_SHAPE;
  if ((long long)kv_stride_tokens < (long long)P + N) return TV_ERR_SHAPE;
  if ((long long)B * Hkv > 65535LL * 65535LL) return TV_ERR_SHAPE;
  if (!(scale >= 0.f) || isinf(scale)) return TV_ERR_VALUE;
  if (scale == 0.f) scale = 1.f / sqrtf((float)D);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return TV_ERR_ALIGN;
  AttnPlan p = attn_plan(B, Hq, Hkv, D, P, N, dtype);
  if (p.tc) {
    if (B > 65535 || Hkv > 65535) return TV_ERR_SHAPE;
    if (workspace && !aligned16(workspace)) return TV_ERR_ALIGN;
    return cuda_status(launch_attn_tc(q, k_cache, v_cache, out, parent, B, Hq, Hkv, D, P, N, kv_stride_tokens, scale,
                                      p, reinterpret_cast<char*>(workspace), ws_bytes, dev_status, st(stream)));
  }
  if ((long long)B * Hq * N / 4 + 1 > 0x7fffffffLL) return TV_ERR_SHAPE;
  return cuda_status(launch_attn_simt(q, k_cache, v_cache, out, parent, B, Hq, Hkv, D, P, N, kv_stride_tokens, scale,
                                      dtype, dev_status, st(stream)));
}

tv_status tv_tree_attention_plan(int B, int Hq, int Hkv, int D, int P, int N, tv_dtype dtype, int* kernel,
                                 int* splits) {
  if (!kernel || !splits) return TV_ERR_NULL;
  if (!valid_dtype(dtype)) return TV_ERR_DTYPE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || N < 1 || N > kMaxNodes || P < 0) return TV_ERR_SHAPE;
  AttnPlan p = attn_plan(B, Hq, Hkv, D, P, N, dtype);
  if (!p.tc) {
    *kernel = 0;
    *splits = 1;
    return TV_OK;
  }
  attn_tc_choice(B, Hkv, D, P, N, p, kernel, splits);
  return TV_OK;
}

size_t tv_verify_workspace_size(int B, int N, int V, tv_dtype, int sampling) {
  if (B < 1 || N < 1 || V < 1) return 0;
  return verify_ws_layout(B, N, V, sampling ? 1 : 0, nullptr);
}

static tv_status verify_common_checks(const void* logits, const int32_t* parent, const int32_t* tokens, int B, int N,
                                      int V, tv_dtype dtype, void* ws, size_t ws_bytes, int sampling) {
  if (!logits || !parent || !tokens) return TV_ERR_NULL;
  if (!valid_dtype(dtype)) return TV_ERR_DTYPE;
  if (B < 1 || N < 1 || N > kMaxNodes || V < 1) return TV_ERR_SHAPE;
  const long long rows = (long long)B * N;
  if (rows > kMaxVerifyRows) return TV_ERR_SHAPE;
  if ((long long)N * V > 0x7fffffffLL) return TV_ERR_SHAPE;
  if (!ws || ws_bytes < verify_ws_layout(B, N, V, sampling, nullptr)) return TV_ERR_WORKSPACE;
  if (!aligned16(ws)) return TV_ERR_ALIGN;
  return TV_OK;
}

tv_status tv_verify_greedy(const void* logits, const int32_t* parent, const int32_t* tokens, int B, int N, int V,
                           tv_dtype dtype, int32_t* accepted_nodes, int32_t* accept_len, int32_t* bonus_token,
                           float* p_draft, float* row_lse, int32_t* row_argmax, void* workspace, size_t ws_bytes,
                           int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_verify_greedy");
  if (!accepted_nodes || !accept_len || !bonus_token) return TV_ERR_NULL;
  tv_status s = verify_common_checks(logits, parent, tokens, B, N, V, dtype, workspace, ws_bytes, 0);
  if (s != TV_OK) return s;
  VerifyWs w;
  verify_ws_layout(B, N, V, 0, &w);
  return cuda_status(launch_vocab_pass(logits, nullptr, parent, tokens, B, N, V, dtype, 1.0f,
                                       reinterpret_cast<char*>(workspace), w, accepted_nodes, accept_len, bonus_token,
                                       p_draft, nullptr, row_lse, row_argmax, nullptr, dev_status, 0,
                                       st(stream)));
}

tv_status tv_vocab_stats(const void* logits, const void* draft_logits, const int32_t* parent,
                         const int32_t* tokens, int B, int N, int V, float temperature, tv_dtype dtype,
                         float* row_lse, int32_t* row_argmax, float* p_draft, float* draft_row_lse, float* q_draft,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_vocab_stats");
  if (!draft_logits && (draft_row_lse || q_draft)) return TV_ERR_NULL;
  if (!(temperature > 0.f) || isinf(temperature)) return TV_ERR_VALUE;
  const int two = draft_logits ? 1 : 0;
  tv_status s = verify_common_checks(logits, parent, tokens, B, N, V, dtype, workspace, ws_bytes, two);
  if (s != TV_OK) return s;
  VerifyWs w;
  verify_ws_layout(B, N, V, two, &w);
  return cuda_status(launch_vocab_pass(logits, draft_logits, parent, tokens, B, N, V, dtype, temperature,
                                       reinterpret_cast<char*>(workspace), w, nullptr, nullptr, nullptr, p_draft,
                                       q_draft, row_lse, row_argmax, draft_row_lse, dev_status, two, st(stream)));
}

tv_status tv_verify_sample(const void* target_logits, const void* draft_logits, const int32_t* parent,
                           const int32_t* tokens, int B, int N, int V, float temperature, uint64_t seed,
                           uint64_t round, tv_dtype dtype, int32_t* accepted_nodes, int32_t* accept_len,
                           int32_t* out_token, float* p_draft, float* q_draft, void* workspace, size_t ws_bytes,
                           int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_verify_sample");
  if (!draft_logits || !accepted_nodes || !accept_len || !out_token) return TV_ERR_NULL;
  if (!(temperature > 0.f) || isinf(temperature)) return TV_ERR_VALUE;
  tv_status s = verify_common_checks(target_logits, parent, tokens, B, N, V, dtype, workspace, ws_bytes, 1);
  if (s != TV_OK) return s;
  VerifyWs w;
  verify_ws_layout(B, N, V, 1, &w);
  char* ws = reinterpret_cast<char*>(workspace);
  cudaError_t e = launch_vocab_pass(target_logits, draft_logits, parent, tokens, B, N, V, dtype, temperature, ws, w,
                                    nullptr, nullptr, nullptr, p_draft, q_draft, nullptr, nullptr, nullptr,
                                    dev_status, 1, st(stream));
  if (e != cudaSuccess) return TV_ERR_CUDA;
  return cuda_status(launch_sample_walk(target_logits, draft_logits, parent, tokens, B, N, V, dtype, temperature,
                                        seed, round, ws, w, accepted_nodes, accept_len, out_token, dev_status,
                                        st(stream)));
}

tv_status tv_commit_accepted_kv(void* k_cache, void* v_cache, const int32_t* accepted_nodes,
                                const int32_t* accept_len, int B, int Hkv, int D, int P, int N, int kv_stride_tokens,
                                tv_dtype dtype, int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_commit_accepted_kv");
  if (!k_cache || !v_cache || !accepted_nodes || !accept_len) return TV_ERR_NULL;
  if (!valid_dtype(dtype)) return TV_ERR_DTYPE;
  if (B < 1 || Hkv < 1 || D < 1 || P < 0 || N < 1 || N > kMaxNodes) return TV_ERR_SHAPE;
  if ((long long)kv_stride_tokens < (long long)P + N) return TV_ERR_SHAPE;
  const long long row_bytes = (long long)D * (dtype == TV_BF16 ? 2 : 4);
  if (row_bytes % 16) return TV_ERR_ALIGN;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return TV_ERR_ALIGN;
  if ((long long)B * Hkv * 2 * (row_bytes / 16) > 0x7fffffffLL * 256) return TV_ERR_SHAPE;
  return cuda_status(launch_kv_commit(k_cache, v_cache, accepted_nodes, accept_len, B, Hkv, D, P, N,
                                      kv_stride_tokens, dtype, dev_status, st(stream)));
}

tv_status tv_frontier_topw(const float* scores, const int32_t* count, int B, int C, int W, int32_t* out_idx,
                           int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_frontier_topw");
  if (!scores || !count || !out_idx) return TV_ERR_NULL;
  if (B < 1 || C < 1 || C > 4096 || W < 1 || W > C) return TV_ERR_SHAPE;
  return cuda_status(launch_frontier_topw(scores, count, B, C, W, out_idx, dev_status, st(stream)));
}

size_t tv_expand_workspace_size(int R, int V, int m) { return expand_ws_bytes(R, V, m); }

tv_status tv_expand_children(const void* draft_logits, const float* parent_score, int R, int V, int m,
                             float temperature, tv_dtype dtype, int32_t* child_token, float* child_p,
                             float* child_score, void* workspace, size_t ws_bytes, int32_t* dev_status,
                             tv_stream_t stream) {
  NvtxRange nvtx_range("tv_expand_children");
  if (!draft_logits || !parent_score || !child_token || !child_p || !child_score) return TV_ERR_NULL;
  if (!valid_dtype(dtype)) return TV_ERR_DTYPE;
  if (R < 1 || V < 1 || m < 1 || m > 32) return TV_ERR_SHAPE;
  if ((long long)R * 32 > 0x7fffffffLL) return TV_ERR_SHAPE;
  if (!(temperature > 0.f) || isinf(temperature)) return TV_ERR_VALUE;
  if (!workspace || ws_bytes < expand_ws_bytes(R, V, m)) return TV_ERR_WORKSPACE;
  if (!aligned16(workspace)) return TV_ERR_ALIGN;
  return cuda_status(launch_expand(draft_logits, parent_score, R, V, m, temperature, dtype, child_token, child_p,
                                   child_score, reinterpret_cast<char*>(workspace), dev_status, st(stream)));
}

size_t tv_select_workspace_size(int B, int d, int K, int budget) { return select_ws_bytes(B, d, K, budget); }

tv_status tv_select_subtree(const float* marg, const int32_t* pool_tokens, int B, int d, int K, int budget,
                            const int32_t* root_token, int32_t* parent, int32_t* tokens, int32_t* depth, float* score,
                            int32_t* n_nodes, void* workspace, size_t ws_bytes, int32_t* dev_status,
                            tv_stream_t stream) {
  NvtxRange nvtx_range("tv_select_subtree");
  if (!marg || !pool_tokens || !parent || !tokens || !depth || !score) return TV_ERR_NULL;
  if (B < 1 || d < 1 || d > kMaxDepth || K < 1 || K > kMaxRank || budget < 1 || budget > kMaxBudget)
    return TV_ERR_SHAPE;
  if (ws_bytes < select_ws_bytes(B, d, K, budget)) return TV_ERR_WORKSPACE;
  return cuda_status(launch_select(marg, pool_tokens, B, d, K, budget, root_token, parent, tokens, depth, score,
                                   n_nodes, reinterpret_cast<char*>(workspace), dev_status, 0.f, 0.f, st(stream)));
}

tv_status tv_select_subtree_adaptive(const float* marg, const int32_t* pool_tokens, int B, int d, int K, int budget,
                                     float cost_base, float cost_per_row, const int32_t* root_token, int32_t* parent,
                                     int32_t* tokens, int32_t* depth, float* score, int32_t* n_nodes,
                                     void* workspace, size_t ws_bytes, int32_t* dev_status, tv_stream_t stream) {
  NvtxRange nvtx_range("tv_select_subtree_adaptive");
  if (!marg || !pool_tokens || !parent || !tokens || !depth || !score || !n_nodes) return TV_ERR_NULL;
  if (B < 1 || d < 1 || d > kMaxDepth || K < 1 || K > kMaxRank || budget < 1 || budget > kMaxBudget)
    return TV_ERR_SHAPE;
  if (!(cost_base >= 0.f) || isinf(cost_base) || !(cost_per_row > 0.f) || isinf(cost_per_row)) return TV_ERR_VALUE;
  if (ws_bytes < select_ws_bytes(B, d, K, budget)) return TV_ERR_WORKSPACE;
  return cuda_status(launch_select(marg, pool_tokens, B, d, K, budget, root_token, parent, tokens, depth, score,
                                   n_nodes, reinterpret_cast<char*>(workspace), dev_status, cost_base, cost_per_row,
                                   st(stream)));
}

}  // extern "C"
