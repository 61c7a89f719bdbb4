// Budgeted prefix-closed subtree selection from a block-marginal pool.
//
// TAPS §4.1: d positions x top-K tokens form the candidate tree; §4.2: edge acceptance
// estimates propagate to path-level reach probabilities, and a prefix-closed subtree is
// kept greedily under the verification budget.  TreeGraft §3.1: cumulative path score
// s(v) = product of the edge scores along the root->v path, s(root) = 1.
// Edge score := the child's marginal; s is built with correctly rounded fp32 multiplies
// from the root down, so the result is reproducible bit for bit.
//
// The first budget-1 candidates in the order (s desc, depth asc, rank path asc) are
// found by best-first search over the first-child / next-sibling form of the candidate
// tree, which is heap-ordered in that order.  One warp per sequence: the frontier lives
// in shared memory; every pop is a warp-wide arg-min over the frontier keys.
#include "tv_kernels.cuh"

namespace tv {

// Frontier key, compared lexicographically (k0, k1, k2) ascending:
//   k0 = (~bits(s)) << 32 | depth      (s >= 0, so larger s -> smaller key)
//   k1, k2 = rank path, one byte per level, level 0 in the top byte of k1
struct FrontierSmem {
  uint64_t* k0;
  uint64_t* k1;
  uint64_t* k2;
  int* par;
  float* psc;
};

__device__ __forceinline__ bool key_less(uint64_t a0, uint64_t a1, uint64_t a2, uint64_t b0, uint64_t b1,
                                         uint64_t b2) {
  if (a0 != b0) return a0 < b0;
  if (a1 != b1) return a1 < b1;
  return a2 < b2;
}

__device__ __forceinline__ int path_rank(uint64_t k1, uint64_t k2, int level) {
  return level < 8 ? (int)((k1 >> (8 * (7 - level))) & 0xFF) : (int)((k2 >> (8 * (15 - level))) & 0xFF);
}

__device__ __forceinline__ void path_bump(uint64_t& k1, uint64_t& k2, int level) {
  if (level < 8)
    k1 += 1ull << (8 * (7 - level));
  else
    k2 += 1ull << (8 * (15 - level));
}

__device__ __forceinline__ uint64_t make_k0(float s, int depth) {
  return ((uint64_t)(~__float_as_uint(s)) << 32) | (uint32_t)depth;
}

__global__ void __launch_bounds__(32) select_kernel(const float* __restrict__ marg, const int32_t* __restrict__ ptok,
                                                    int d, int K, int budget, const int32_t* __restrict__ root_token,
                                                    int32_t* out_parent, int32_t* out_tok, int32_t* out_depth,
                                                    float* out_score, int32_t* n_nodes, int32_t* dev_status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int b = blockIdx.x, lane = threadIdx.x;
  const int cap = budget;  // frontier never exceeds 1 + pops <= budget
  uint64_t* k0 = reinterpret_cast<uint64_t*>(smem);
  uint64_t* k1 = k0 + cap;
  uint64_t* k2 = k1 + cap;
  float* sm_marg = reinterpret_cast<float*>(k2 + cap);
  int* sm_tok = reinterpret_cast<int*>(sm_marg + d * K);
  int* par = sm_tok + d * K;
  float* psc = reinterpret_cast<float*>(par + cap);

  const float* mg = marg + (size_t)b * d * K;
  const int32_t* tk = ptok + (size_t)b * d * K;
  int bad = 0;
  for (int i = lane; i < d * K; i += 32) {
    const float m = mg[i];
    sm_marg[i] = m;
    sm_tok[i] = tk[i];
    const bool sorted = (i % K == 0) || !(m > mg[i - 1]);
    if (!(m >= 0.f && m <= 1.f) || !sorted) bad = 1;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_dev_status(dev_status, TV_DEV_BAD_TOKEN);
  __syncwarp();

  int32_t* o_par = out_parent + (size_t)b * budget;
  int32_t* o_tok = out_tok + (size_t)b * budget;
  int32_t* o_dep = out_depth + (size_t)b * budget;
  float* o_sc = out_score + (size_t)b * budget;
  if (lane == 0) {
    o_par[0] = -1;
    o_tok[0] = root_token ? root_token[b] : -1;
    o_dep[0] = 0;
    o_sc[0] = 1.f;
  }
  int F = 0;
  if (d >= 1 && K >= 1 && budget > 1) {
    if (lane == 0) {
      const float s0 = __fmul_rn(1.f, sm_marg[0]);
      k0[0] = make_k0(s0, 1);
      k1[0] = 0;
      k2[0] = 0;
      par[0] = 0;
      psc[0] = 1.f;
    }
    F = 1;
  }
  __syncwarp();
  int n = 1;
  while (F > 0 && n < budget) {
    // warp arg-min over the frontier
    uint64_t b0 = ~0ull, b1 = ~0ull, b2 = ~0ull;
    int bi = -1;
    for (int i = lane; i < F; i += 32) {
      const uint64_t a0 = k0[i], a1 = k1[i], a2 = k2[i];
      if (bi < 0 || key_less(a0, a1, a2, b0, b1, b2)) {
        b0 = a0;
        b1 = a1;
        b2 = a2;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t c0 = __shfl_xor_sync(0xffffffffu, b0, o);
      const uint64_t c1 = __shfl_xor_sync(0xffffffffu, b1, o);
      const uint64_t c2 = __shfl_xor_sync(0xffffffffu, b2, o);
      const int ci = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ci >= 0 && (bi < 0 || key_less(c0, c1, c2, b0, b1, b2))) {
        b0 = c0;
        b1 = c1;
        b2 = c2;
        bi = ci;
      }
    }
    if (lane == 0) {
      const int dep = (int)(b0 & 0xFFFFFFFFu);
      const float s = __uint_as_float(~(uint32_t)(b0 >> 32));
      const int p = par[bi];
      const float ps = psc[bi];
      const int r = path_rank(b1, b2, dep - 1);
      o_par[n] = p;
      o_tok[n] = sm_tok[(dep - 1) * K + r];
      o_dep[n] = dep;
      o_sc[n] = s;
      // remove the popped entry
      const int last = F - 1;
      k0[bi] = k0[last];
      k1[bi] = k1[last];
      k2[bi] = k2[last];
      par[bi] = par[last];
      psc[bi] = psc[last];
      int f = last;
      if (dep < d) {  // first child: rank 0 at the next position
        const float sc = __fmul_rn(s, sm_marg[dep * K + 0]);
        k0[f] = make_k0(sc, dep + 1);
        k1[f] = b1;
        k2[f] = b2;
        par[f] = n;
        psc[f] = s;
        ++f;
      }
      if (r + 1 < K) {  // next sibling under the same parent
        const float ss = __fmul_rn(ps, sm_marg[(dep - 1) * K + r + 1]);
        uint64_t n1 = b1, n2 = b2;
        path_bump(n1, n2, dep - 1);
        k0[f] = make_k0(ss, dep);
        k1[f] = n1;
        k2[f] = n2;
        par[f] = p;
        psc[f] = ps;
        ++f;
      }
      F = f;
    }
    F = __shfl_sync(0xffffffffu, F, 0);
    ++n;
    __syncwarp();
  }
  for (int j = n + lane; j < budget; j += 32) {
    o_par[j] = -1;
    o_tok[j] = -1;
    o_dep[j] = -1;
    o_sc[j] = 0.f;
  }
  if (lane == 0 && n_nodes) n_nodes[b] = n;
}

static size_t select_smem_bytes(int d, int K, int budget) {
  return (size_t)budget * (3 * 8 + 4 + 4) + (size_t)d * K * 8;
}

size_t select_ws_bytes(int, int, int, int) { return 0; }

cudaError_t launch_select(const float* marg, const int32_t* ptok, int B, int d, int K, int budget,
                          const int32_t* root_token, int32_t* parent, int32_t* tokens, int32_t* depth,
                          float* score, int32_t* n_nodes, char*, int32_t* dev_status, cudaStream_t stream) {
  const size_t smem = select_smem_bytes(d, K, budget);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  select_kernel<<<B, 32, smem, stream>>>(marg, ptok, d, K, budget, root_token, parent, tokens, depth, score,
                                         n_nodes, dev_status);
  return cudaGetLastError();
}

}  // namespace tv
