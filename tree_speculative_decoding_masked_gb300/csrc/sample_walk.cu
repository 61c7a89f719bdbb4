// Stochastic acceptance walk down the draft tree (one CTA of 1024 threads per sequence).
//
// Speculative-decoding blog, "acceptance probability for sampling": draft token t of
// node c is kept with probability min(1, p(t)/q(t)); "how to correct after a
// rejection": the replacement is drawn from (p - q)+ / sum (p - q)+.  With several
// drafted children per node they are tried in ascending node index; after rejecting
// t_k the target side moves to the normalised residual and the draft side drops t_k and
// renormalises (the drafts at one node are distinct tokens).  Each residual needs one
// pass over the vocabulary (its normaliser Z); the final draw needs one more pass
// (an inverse-CDF scan).  Sums run in fp64.
#include "philox.cuh"
#include "tv_kernels.cuh"

namespace tv {

constexpr int kWalkThreads = 1024;
constexpr int kMaxRejections = kMaxNodes;  // a node has fewer than N children

struct WalkArgs {
  const void* target;
  const void* draft;
  const int32_t* parent;
  const int32_t* tokens;
  int N, V;
  float c2;
  uint64_t seed, round;
  const float* lse2;
  const float* lse2_q;
  const float* pc;
  const float* qc;
  int32_t* accepted;
  int32_t* accept_len;
  int32_t* out_token;
  int32_t* dev_status;
};

template <typename T>
__device__ __forceinline__ float ld_logit(const void* base, size_t i) {
  if constexpr (sizeof(T) == 2)
    return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
  else
    return reinterpret_cast<const float*>(base)[i];
}

// State of the residual recursion at one node after `nrej` rejections.
struct Residual {
  int nrej;
  int tok[kMaxRejections];     // rejected tokens t_1..t_nrej
  float invz[kMaxRejections];  // 1 / Z_j (0 when Z_j == 0: keep P_j)
  float invd[kMaxRejections + 1];  // 1 / D_j, D_j = 1 - sum_{i<j} q(t_i)  (0 when nothing left)
};

// P_{n+1}(v), Q_{n+1}(v) for n = r.nrej rejections, from p(v), q(v) at the node.
__device__ __forceinline__ void eval_pq(const Residual& r, int v, float p, float q, float& P, float& Q) {
  P = p;
  bool removed = false;
  for (int j = 0; j < r.nrej; ++j) {
    const float Qj = removed ? 0.f : q * r.invd[j];
    if (r.invz[j] > 0.f) P = fmaxf(P - Qj, 0.f) * r.invz[j];
    removed = removed || (v == r.tok[j]);
  }
  Q = removed ? 0.f : q * r.invd[r.nrej];
}

__device__ double block_sum_d(double v, double* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) red[wid] = v;
  __syncthreads();
  if (wid == 0) {
    double x = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0;
    x = warp_sum_d(x);
    if (lane == 0) red[32] = x;
  }
  __syncthreads();
  double r = red[32];
  __syncthreads();
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kWalkThreads) sample_walk_kernel(WalkArgs a) {
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_kids[kMaxNodes];
  __shared__ int s_wcnt[32];
  __shared__ int s_nkids, s_bad, s_found;
  __shared__ double red[33];
  __shared__ Residual res;
  __shared__ int s_dec;  // broadcast of a decision
  const int b = blockIdx.x;
  const int N = a.N, V = a.V;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int c = tid; c < N; c += blockDim.x) {
    const int p = a.parent[(size_t)b * N + c];
    const int t = a.tokens[(size_t)b * N + c];
    s_par[c] = p;
    s_tok[c] = t;
    const bool ok = (c == 0) ? (p == -1) : (p >= 0 && p < c);
    if (!ok) atomicOr(&s_bad, TV_DEV_BAD_TREE);
    if (c > 0 && (t < 0 || t >= V)) atomicOr(&s_bad, TV_DEV_BAD_TOKEN);
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      set_dev_status(a.dev_status, s_bad);
      a.accept_len[b] = 0;
      a.out_token[b] = -1;
    }
    for (int j = tid; j < N; j += blockDim.x) a.accepted[(size_t)b * N + j] = -1;
    return;
  }
  int u = 0, len = 0;
  for (;;) {
    // ---- children of u in ascending node index
    {
      int c = tid;  // N <= 1024 = blockDim
      const bool hit = c < N && c > u && s_par[c] == u;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (lane == 0) s_wcnt[wid] = __popc(m);
      __syncthreads();
      if (wid == 0) {
        int x = s_wcnt[lane];
        int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        s_wcnt[lane] = incl - x;
        if (lane == 31) s_nkids = incl;
      }
      __syncthreads();
      if (hit) s_kids[s_wcnt[wid] + __popc(m & ((1u << lane) - 1u))] = c;
      if (tid == 0) {
        res.nrej = 0;
        res.invd[0] = 1.f;
        s_found = -1;
      }
      __syncthreads();
    }
    const int m = s_nkids;
    const size_t rowp = ((size_t)b * N + u) * (size_t)V;
    const float l2p = a.lse2[(size_t)b * N + u];
    const float l2q = a.lse2_q[(size_t)b * N + u];
    for (int k = 1; k <= m; ++k) {
      const int c = s_kids[k - 1];
      if (tid == 0) {
        const int t = s_tok[c];
        float pt, qt;
        if (res.nrej == 0) {
          pt = a.pc[(size_t)b * N + c];
          qt = a.qc[(size_t)b * N + c];
        } else {
          const float p0 = exp2f(fmaf(ld_logit<T>(a.target, rowp + t), a.c2, -l2p));
          const float q0 = exp2f(fmaf(ld_logit<T>(a.draft, rowp + t), a.c2, -l2q));
          eval_pq(res, t, p0, q0, pt, qt);
        }
        const float r = philox_uniform(a.seed, a.round, b, u, k, 0);
        const float alpha = qt > 0.f ? fminf(1.f, __fdiv_rn(pt, qt)) : (pt > 0.f ? 1.f : 0.f);
        s_dec = (r < alpha) ? 1 : 0;
        if (s_dec) s_found = c;
      }
      __syncthreads();
      if (s_dec) break;
      // rejection of t_k: Z = sum_v (P(v) - Q(v))+ with the current (P, Q)
      double zs = 0.0;
      for (int v = tid; v < V; v += blockDim.x) {
        const float p0 = exp2f(fmaf(ld_logit<T>(a.target, rowp + v), a.c2, -l2p));
        const float q0 = exp2f(fmaf(ld_logit<T>(a.draft, rowp + v), a.c2, -l2q));
        float P, Q;
        eval_pq(res, v, p0, q0, P, Q);
        zs += (double)fmaxf(P - Q, 0.f);
      }
      const double z = block_sum_d(zs, red);
      if (tid == 0) {
        const int j = res.nrej;
        const int t = s_tok[c];
        const float q0 = exp2f(fmaf(ld_logit<T>(a.draft, rowp + t), a.c2, -l2q));
        res.tok[j] = t;
        res.invz[j] = z > 0.0 ? (float)(1.0 / z) : 0.f;
        const float dprev = res.invd[j] > 0.f ? 1.f / res.invd[j] : 0.f;
        const float dnext = dprev - q0;
        res.invd[j + 1] = dnext > 0.f ? 1.f / dnext : 0.f;
        res.nrej = j + 1;
      }
      __syncthreads();
    }
    if (s_found >= 0) {
      const int c = s_found;
      if (tid == 0) a.accepted[(size_t)b * N + len] = c;
      ++len;
      u = c;
      __syncthreads();
      continue;
    }
    // ---- final draw from the current P by inverse CDF (blocked fp64 scan)
    const int per = (V + blockDim.x - 1) / blockDim.x;
    const int v0 = min(V, tid * per), v1 = min(V, v0 + per);
    double loc = 0.0;
    for (int v = v0; v < v1; ++v) {
      const float p0 = exp2f(fmaf(ld_logit<T>(a.target, rowp + v), a.c2, -l2p));
      const float q0 = res.nrej ? exp2f(fmaf(ld_logit<T>(a.draft, rowp + v), a.c2, -l2q)) : 0.f;
      float P, Q;
      eval_pq(res, v, p0, q0, P, Q);
      loc += (double)P;
    }
    // exclusive scan of `loc` across the block
    double incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) red[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      double x = red[lane];
      double xi = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        double y = __shfl_up_sync(0xffffffffu, xi, o);
        if (lane >= o) xi += y;
      }
      red[lane] = xi - x;
      if (lane == 31) red[32] = xi;
    }
    __syncthreads();
    const double excl = red[wid] + (incl - loc);
    const double total = red[32];
    const float r = philox_uniform(a.seed, a.round, b, u, 0, 1);
    const double target = (double)r * total;
    if (tid == 0) s_found = 0x7fffffff;
    __syncthreads();
    if (target >= excl && target < excl + loc) {
      // this thread's slice holds the crossing: smallest v with target < prefix(v)
      double run = excl;
      int pick = -1, last_pos = -1;
      for (int v = v0; v < v1; ++v) {
        const float p0 = exp2f(fmaf(ld_logit<T>(a.target, rowp + v), a.c2, -l2p));
        const float q0 = res.nrej ? exp2f(fmaf(ld_logit<T>(a.draft, rowp + v), a.c2, -l2q)) : 0.f;
        float P, Q;
        eval_pq(res, v, p0, q0, P, Q);
        if (P > 0.f) last_pos = v;
        run += (double)P;
        if (target < run) {
          pick = v;
          break;
        }
      }
      if (pick < 0) pick = last_pos;
      if (pick >= 0) atomicMin(&s_found, pick);
    }
    __syncthreads();
    if (tid == 0 && s_found == 0x7fffffff) s_found = V - 1;
    __syncthreads();
    if (tid == 0) {
      a.out_token[b] = s_found;
      a.accept_len[b] = len;
    }
    for (int j = len + tid; j < N; j += blockDim.x) a.accepted[(size_t)b * N + j] = -1;
    return;
  }
}

cudaError_t launch_sample_walk(const void* target, const void* draft, const int32_t* parent,
                               const int32_t* tokens, int B, int N, int V, tv_dtype dtype, float temperature,
                               uint64_t seed, uint64_t round, char* ws, const VerifyWs& w,
                               int32_t* accepted, int32_t* accept_len, int32_t* out_token,
                               int32_t* dev_status, cudaStream_t stream) {
  WalkArgs a;
  a.target = target;
  a.draft = draft;
  a.parent = parent;
  a.tokens = tokens;
  a.N = N;
  a.V = V;
  a.c2 = kLog2e / temperature;
  a.seed = seed;
  a.round = round;
  a.lse2 = reinterpret_cast<const float*>(ws + w.lse2);
  a.lse2_q = reinterpret_cast<const float*>(ws + w.lse2_q);
  a.pc = reinterpret_cast<const float*>(ws + w.pc);
  a.qc = reinterpret_cast<const float*>(ws + w.qc);
  a.accepted = accepted;
  a.accept_len = accept_len;
  a.out_token = out_token;
  a.dev_status = dev_status;
  if (dtype == TV_BF16)
    sample_walk_kernel<uint16_t><<<B, kWalkThreads, 0, stream>>>(a);
  else
    sample_walk_kernel<float><<<B, kWalkThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace tv
