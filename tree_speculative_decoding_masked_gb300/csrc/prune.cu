// Width and depth control of a draft tree, one CTA per sequence, one thread per node.
//
// PTD §3.1 "overhead constraints": a cap on the children of every parent (the most
// confident children stay) and sliding-window stepping - while the kept tree is deeper
// than the threshold, the root's earliest-added kept child becomes the root and the
// other branches are pruned.  Nodes are numbered in the order they were added, so
// "earliest" is the lowest index; the survivors are renumbered in that order.
#include "tv_kernels.cuh"

namespace tv {

constexpr int kPruneThreads = 1024;  // one thread per node (N <= kMaxNodes)

__global__ void __launch_bounds__(kPruneThreads) prune_kernel(const int32_t* parent, const float* conf, int N,
                                                            int max_children, int depth_limit, int32_t* old_to_new,
                                                            int32_t* new_parent, int32_t* n_kept, int32_t* new_root,
                                                            int32_t* dev_status) {
  __shared__ int s_par[kMaxNodes];
  __shared__ float s_conf[kMaxNodes];
  __shared__ int s_dep[kMaxNodes];
  __shared__ int s_keep[kMaxNodes];
  __shared__ int s_md[kMaxNodes];  // deepest kept descendant's depth (absolute)
  __shared__ int s_fc[kMaxNodes];  // lowest-index kept child
  __shared__ int s_new[kMaxNodes];
  __shared__ int s_wsum[32];
  __shared__ int s_root, s_bad;
  const int b = blockIdx.x, v = threadIdx.x;
  const bool node = v < N;
  if (v == 0) s_bad = 0;
  if (node) {
    const int p = parent[(size_t)b * N + v];
    s_par[v] = p;
    s_conf[v] = conf[(size_t)b * N + v];
    s_md[v] = -1;
    s_fc[v] = 0x7fffffff;
  }
  __syncthreads();
  if (node) {
    const int p = s_par[v];
    if (!((v == 0) ? (p == -1) : (p >= 0 && p < v))) atomicOr(&s_bad, TV_DEV_BAD_TREE);
  }
  __syncthreads();
  if (s_bad) {
    if (v == 0) {
      set_dev_status(dev_status, s_bad);
      n_kept[b] = 0;
      new_root[b] = -1;
    }
    if (node) {
      old_to_new[(size_t)b * N + v] = -1;
      new_parent[(size_t)b * N + v] = -1;
    }
    return;
  }
  // depth, and the width rule: rank among siblings by (confidence desc, index asc)
  int keep0 = 1, dep = 0;
  if (node && v > 0) {
    for (int a = s_par[v]; a >= 0; a = s_par[a]) ++dep;
    const int p = s_par[v];
    const float c = s_conf[v];
    int rank = 0;
    for (int j = p + 1; j < N; ++j)  // siblings have larger indices than their parent
      if (s_par[j] == p && (s_conf[j] > c || (s_conf[j] == c && j < v))) ++rank;
    keep0 = rank < max_children;
  }
  if (node) {
    s_dep[v] = dep;
    s_keep[v] = keep0;
  }
  __syncthreads();
  // a node stays only if every ancestor passed the width rule
  int kept = 0;
  if (node) {
    kept = s_keep[v];
    for (int a = s_par[v]; a >= 0 && kept; a = s_par[a]) kept = s_keep[a];
  }
  __syncthreads();
  if (node) s_keep[v] = kept;
  __syncthreads();
  if (node && kept) {
    for (int a = v; a >= 0; a = s_par[a]) atomicMax(&s_md[a], dep);
    if (v > 0) atomicMin(&s_fc[s_par[v]], v);
  }
  __syncthreads();
  if (v == 0) {
    int r = 0;
    while (s_md[r] - s_dep[r] > depth_limit && s_fc[r] != 0x7fffffff) r = s_fc[r];
    s_root = r;
  }
  __syncthreads();
  const int root = s_root, rdep = s_dep[root];
  if (node && kept) {  // inside the new root's subtree?
    int a = v;
    while (s_dep[a] > rdep) a = s_par[a];
    kept = a == root;
  }
  // compaction in index order: block exclusive scan of the keep flags
  const int lane = v & 31, w = v >> 5;
  const int flag = node && kept ? 1 : 0;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) s_wsum[w] = __popc(bal);
  __syncthreads();
  if (w == 0) {
    const int x = s_wsum[lane];
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    s_wsum[lane] = incl - x;
    if (lane == 31) s_md[0] = incl;  // total (s_md is no longer needed)
  }
  __syncthreads();
  const int idx = s_wsum[w] + __popc(bal & ((1u << lane) - 1u));
  if (node) s_new[v] = flag ? idx : -1;
  __syncthreads();
  const int total = s_md[0];
  if (node) {
    old_to_new[(size_t)b * N + v] = s_new[v];
    if (flag) new_parent[(size_t)b * N + idx] = v == root ? -1 : s_new[s_par[v]];
  }
  for (int i = total + v; i < N; i += blockDim.x) new_parent[(size_t)b * N + i] = -1;
  if (v == 0) {
    n_kept[b] = total;
    new_root[b] = root;
  }
}

cudaError_t launch_prune(const int32_t* parent, const float* conf, int B, int N, int max_children, int depth_limit,
                         int32_t* old_to_new, int32_t* new_parent, int32_t* n_kept, int32_t* new_root,
                         int32_t* dev_status, cudaStream_t stream) {
  prune_kernel<<<B, kPruneThreads, 0, stream>>>(parent, conf, N, max_children, depth_limit, old_to_new, new_parent,
                                               n_kept, new_root, dev_status);
  return cudaGetLastError();
}

}  // namespace tv
