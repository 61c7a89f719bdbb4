// Internal declarations shared between the kernel files and the C-ABI layer.
#pragma once

#include "tv_common.cuh"

namespace tv {

constexpr int kMaxNodes = 1024;  // N limit (tree nodes per sequence, root included)
constexpr int kMaxDepth = 16;    // selection pool depth d
constexpr int kMaxRank = 256;    // selection pool width K
constexpr int kMaxBudget = 4096; // selection budget (rows)

// ---- verify (vocab pass + walks)
struct VerifyWs {
  int splits;  // partial slots per row
  size_t row_cnt, seq_cnt, part, part_q, lse2, lse2_q, xc, pc, qc, yc, total;
};
constexpr long long kMaxVerifyRows = 131072;  // B * N limit of the verify calls
int verify_slots_per_row(int rows);
size_t verify_ws_layout(int B, int N, int V, int sampling, VerifyWs* w);
cudaError_t launch_vocab_pass(const void* logits, const void* draft, const int32_t* parent,
                              const int32_t* tokens, int B, int N, int V, tv_dtype dtype, float temperature,
                              char* ws, const VerifyWs& w, int32_t* accepted, int32_t* accept_len,
                              int32_t* bonus, float* p_draft, float* q_draft, float* row_lse,
                              int32_t* row_argmax, float* row_lse_q, int32_t* dev_status, int sampling,
                              cudaStream_t stream);
cudaError_t launch_sample_walk(const void* target, const void* draft, const int32_t* parent,
                               const int32_t* tokens, int B, int N, int V, tv_dtype dtype, float temperature,
                               uint64_t seed, uint64_t round, char* ws, const VerifyWs& w,
                               int32_t* accepted, int32_t* accept_len, int32_t* out_token,
                               int32_t* dev_status, cudaStream_t stream);

// ---- Philox4x32-10 words (the sampling walk's generator)
cudaError_t launch_philox_words(uint64_t seed, const uint32_t* ctr, int n, uint32_t* out, cudaStream_t stream);

// ---- bounded-wait self-test
cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t* dev_status, cudaStream_t stream);

// ---- tree prep
cudaError_t launch_tree_prep(const int32_t* parent, int B, int N, int P, int32_t* depth, int32_t* pos,
                             uint32_t* anc_mask, int32_t* child_off, int32_t* child_idx,
                             int32_t* dev_status, cudaStream_t stream);

// ---- accepted-path KV commit
cudaError_t launch_kv_commit(void* k_cache, void* v_cache, const int32_t* accepted, const int32_t* accept_len,
                             int B, int Hkv, int D, int P, int N, int S, tv_dtype dtype, int32_t* dev_status,
                             cudaStream_t stream);

// ---- single-drafter expansion step
cudaError_t launch_frontier_topw(const float* scores, const int32_t* count, int B, int C, int W, int32_t* out_idx,
                                 int32_t* dev_status, cudaStream_t stream);
size_t expand_ws_bytes(int R, int V, int m);
cudaError_t launch_expand(const void* logits, const float* parent_score, int R, int V, int m, float temperature,
                          tv_dtype dtype, int32_t* child_token, float* child_p, float* child_score, char* ws,
                          int32_t* dev_status, cudaStream_t stream);

// ---- width / depth control
cudaError_t launch_prune(const int32_t* parent, const float* conf, int B, int N, int max_children, int depth_limit,
                         int32_t* old_to_new, int32_t* new_parent, int32_t* n_kept, int32_t* new_root,
                         int32_t* dev_status, cudaStream_t stream);

// ---- SM shares set by tv_set_sm_partition (0 = the whole device)
int sm_share_verify();
int sm_share_attention();
// ---- tensor-core attention kernel set by tv_set_attention_variant (0 = automatic)
int attention_variant();
// ---- forced KV split count set by tv_set_attention_splits (0 = automatic)
int attention_splits();

// ---- selection
size_t select_ws_bytes(int B, int d, int K, int budget);
cudaError_t launch_select(const float* marg, const int32_t* ptok, int B, int d, int K, int budget,
                          const int32_t* root_token, int32_t* parent, int32_t* tokens, int32_t* depth,
                          float* score, int32_t* n_nodes, char* ws, int32_t* dev_status, float cost_base,
                          float cost_per_row, cudaStream_t stream);

// ---- attention
struct AttnPlan {
  bool tc;        // tensor-core (tcgen05) kernel
  int nt;         // nodes per 128-row tile (tc)
  int mtiles;     // row tiles per (b, kv head)
  size_t total;   // workspace bytes (the persistent schedule's partials; 0 for the others)
};
AttnPlan attn_plan(int B, int Hq, int Hkv, int D, int P, int N, tv_dtype dtype);
cudaError_t launch_attn_simt(const void* q, const void* k, const void* v, void* out, const int32_t* parent,
                             int B, int Hq, int Hkv, int D, int P, int N, int S, float scale, tv_dtype dtype,
                             int32_t* dev_status, cudaStream_t stream);
// kernel variant (1 attn_tc_kernel, 2 attn_pair_kernel, 3 attn_pair2_kernel, 4
// attn_stream_kernel) and KV splits the next launch would use
void attn_tc_choice(int B, int Hkv, int D, int P, int N, const AttnPlan& plan, int* var, int* splits);
cudaError_t launch_attn_tc(const void* q, const void* k, const void* v, void* out, const int32_t* parent,
                           int B, int Hq, int Hkv, int D, int P, int N, int S, float scale, const AttnPlan& plan,
                           char* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream);

}  // namespace tv
