// Stochastic acceptance walk down the draft tree (one cluster of CTAs per sequence).
//
// Speculative-decoding blog, "acceptance probability for sampling": draft token t of
// node c is kept with probability min(1, p(t)/q(t)); "how to correct after a
// rejection": the replacement is drawn from (p - q)+ / sum (p - q)+.  With several
// drafted children per node they are tried in ascending node index; after rejecting
// t_k the target side moves to the normalised residual and the draft side drops t_k and
// renormalises (the drafts at one node are distinct tokens).  Each residual needs one
// pass over the vocabulary (its normaliser Z); the final draw needs one more pass
// (an inverse-CDF scan).
//
// Every CTA of the cluster runs the same control flow (same tree, same Philox draws, same
// sums, hence the same decisions) and takes an equal share of the vocabulary in each
// pass.  Where its share fits in shared memory, a CTA loads the node's target and draft
// rows once, as p(v) and q(v), at the node's first full pass and keeps the residual
// P_n(v) there, updated in place after each rejection with the same float operations as
// replaying the recursion from p and q (a rejected token is removed by zeroing its q);
// otherwise every pass reads the rows again and replays the recursion.
// Sums are exact: each term in [0, 1] is rounded once to a multiple of 2^-56 and added as
// a 64-bit integer, so a total does not depend on the order of the additions and every
// CTA, after reading the others' partial sums through distributed shared memory, holds
// the same value.
#include <atomic>

#include "philox.cuh"
#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

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
  int csize;   // CTAs per cluster (one cluster per sequence)
  int cached;  // the share of a row fits the dynamic shared memory (p, q as fp32)
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

constexpr int kWalkClusterMax = 16;  // CTAs per sequence where the device allows it, else 8
constexpr int kBatch = 5;            // vocabulary elements per thread whose loads are issued together
constexpr int kWalkDynCap = 180 * 1024;  // dynamic shared memory for the cached rows

// x * 2^56 rounded to the nearest integer (ties to even), for x in [0, 1], with two
// 32-bit conversions: t = x * 2^24 and its integer part h are exact, so x * 2^56 =
// h * 2^32 + (t - h) * 2^32 and only the second term needs rounding.  (The float to
// 64-bit integer conversion instruction is slow on this part; this form gives the same
// value for every float in [0, 1].)
__device__ __forceinline__ unsigned long long to_fix(float x) {
  const float t = __fmul_rn(x, 0x1p24f);
  const float h = floorf(t);
  const uint32_t lo = __float2uint_rn(__fmul_rn(__fsub_rn(t, h), 0x1p32f));
  return ((unsigned long long)__float2uint_rz(h) << 32) + lo;
}

__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kWalkThreads) sample_walk_kernel(WalkArgs a) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_kids[kMaxNodes];
  __shared__ int s_wcnt[32];
  __shared__ int s_nkids, s_bad, s_found;
  __shared__ unsigned long long red[33];
  __shared__ unsigned long long s_part[2];  // this CTA's sum in a pass (alternating slots)
  __shared__ unsigned long long s_sum[2];   // cluster total and the sum of the lower ranks
  __shared__ float s_pc[kMaxNodes], s_qc[kMaxNodes], s_l2p[kMaxNodes], s_l2q[kMaxNodes];
  __shared__ Residual res;
  __shared__ int s_dec;  // broadcast of a decision
  const uint32_t crank = cluster_rank();
  const int csize = a.csize;
  const int b = blockIdx.x / csize;
  const int N = a.N, V = a.V;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // this CTA's share of the vocabulary in every pass
  const int span = (V + csize - 1) / csize;
  const int vlo = min(V, (int)crank * span), vhi = min(V, vlo + span);
  int npass = 0;
  // cached rows: sP[i] = P_n(vlo + i) at the current node, sQ[i] = q(vlo + i) (0 once the
  // token was rejected there)
  extern __shared__ __align__(16) float walk_dyn[];
  float* sP = walk_dyn;
  float* sQ = walk_dyn + ((span + 3) & ~3);
  const bool cached = a.cached != 0;
  int loaded_u = -1;   // node whose p (and q) are in sP / sQ
  bool loaded_q = false;
  // the last rejection's update of sP / sQ, applied by the next sweep over them:
  // P = (P - q / D_j)+ / Z_j where Z_j > 0, then q(t_j) = 0
  bool pend = false;
  float pend_invz = 0.f, pend_invd = 0.f;
  int pend_tok = -1;
  // Sum of `mine` over the cluster: every CTA gets the same total; *below = the sum over
  // the lower-ranked CTAs
  auto cluster_total = [&](unsigned long long mine, unsigned long long* below) {
    const int slot = npass & 1;
    if (tid == 0) s_part[slot] = mine;
    ptx::cluster_sync();
    if (tid < 32) {  // lane r reads CTA r's partial; the 16 remote loads overlap
      const uint32_t r = (uint32_t)lane;
      const unsigned long long x =
          r < (uint32_t)csize ? ld_cluster_u64(ptx::map_cluster(ptx::smem_addr(&s_part[slot]), r)) : 0ull;
      unsigned long long tot = x, lower = r < crank ? x : 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        lower += __shfl_xor_sync(0xffffffffu, lower, o);
      }
      if (lane == 0) {
        s_sum[0] = tot;
        s_sum[1] = lower;
      }
    }
    __syncthreads();
    const unsigned long long tot = s_sum[0];
    *below = s_sum[1];
    __syncthreads();
    ++npass;
    return tot;
  };
  // p(v) (and q(v) when `with_q`) of this CTA's share of node u's rows into sP / sQ:
  // 16-byte loads, two per array and thread in flight, where the share is 16-byte aligned
  // (else element loads)
  auto load_rows = [&](int node, bool with_q) {
    const size_t row = ((size_t)b * N + node) * (size_t)V;
    const float l2p = s_l2p[node], l2q = s_l2q[node];
    const int n = vhi - vlo;
    constexpr int kE = 16 / (int)sizeof(T);  // elements per 16-byte vector
    const bool vec = (row + (size_t)vlo) % kE == 0 &&
                     ((reinterpret_cast<uintptr_t>(a.target) | reinterpret_cast<uintptr_t>(a.draft)) & 15u) == 0;
    int start = 0;
    if (vec) {
      const int nv = n / kE;
      const uint4* X = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.target) + row + vlo);
      const uint4* Y = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.draft) + row + vlo);
      for (int j0 = tid; j0 < nv; j0 += 2 * (int)blockDim.x) {
        uint4 xv[2], yv[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = j0 + k * (int)blockDim.x;
          xv[k] = j < nv ? __ldg(X + j) : make_uint4(0u, 0u, 0u, 0u);
          yv[k] = (with_q && j < nv) ? __ldg(Y + j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = j0 + k * (int)blockDim.x;
          if (j >= nv) continue;
          const uint32_t xw[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
          const uint32_t yw[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
#pragma unroll
          for (int e = 0; e < kE; ++e) {
            float xf, yf;
            if constexpr (sizeof(T) == 2) {  // element e: half e & 1 of word e / 2, low half first
              xf = __uint_as_float((e & 1) ? (xw[e >> 1] & 0xFFFF0000u) : (xw[e >> 1] << 16));
              yf = __uint_as_float((e & 1) ? (yw[e >> 1] & 0xFFFF0000u) : (yw[e >> 1] << 16));
            } else {
              xf = __uint_as_float(xw[e]);
              yf = __uint_as_float(yw[e]);
            }
            sP[j * kE + e] = ptx::ex2(fmaf(xf, a.c2, -l2p));
            if (with_q) sQ[j * kE + e] = ptx::ex2(fmaf(yf, a.c2, -l2q));
          }
        }
      }
      start = nv * kE;
    }
    for (int i = start + tid; i < n; i += blockDim.x) {
      sP[i] = ptx::ex2(fmaf(ld_logit<T>(a.target, row + vlo + i), a.c2, -l2p));
      if (with_q) sQ[i] = ptx::ex2(fmaf(ld_logit<T>(a.draft, row + vlo + i), a.c2, -l2q));
    }
    __syncthreads();
    loaded_u = node;
    loaded_q = with_q;
    pend = false;
  };
  // element i of the cached rows with the pending update applied (and stored back)
  auto cur_pq = [&](int i, float& P, float& q) {
    P = sP[i];
    q = sQ[i];
    if (pend) {
      if (pend_invz > 0.f) P = fmaxf(P - q * pend_invd, 0.f) * pend_invz;
      if (vlo + i == pend_tok) q = 0.f;
      sP[i] = P;
      sQ[i] = q;
    }
  };
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int c = tid; c < N; c += blockDim.x) {
    const int p = a.parent[(size_t)b * N + c];
    const int t = a.tokens[(size_t)b * N + c];
    s_par[c] = p;
    s_tok[c] = t;
    // per-node inputs of the decisions, in the same round trip
    s_pc[c] = a.pc[(size_t)b * N + c];
    s_qc[c] = a.qc[(size_t)b * N + c];
    s_l2p[c] = a.lse2[(size_t)b * N + c];
    s_l2q[c] = a.lse2_q[(size_t)b * N + c];
    // padding rows of a ragged batch (parent -1 after the last node) are no drafts
    const bool ok = (c == 0) ? (p == -1) : (p == -1 || (p >= 0 && p < c));
    if (!ok) atomicOr(&s_bad, TV_DEV_BAD_TREE);
    if (c > 0 && p != -1 && (t < 0 || t >= V)) atomicOr(&s_bad, TV_DEV_BAD_TOKEN);
  }
  __syncthreads();
  for (int c = 2 + tid; c < N; c += blockDim.x)  // no active row after a padding row
    if (s_par[c] != -1 && s_par[c - 1] == -1) atomicOr(&s_bad, TV_DEV_BAD_TREE);
  __syncthreads();
  if (s_bad) {
    if (crank == 0) {
      if (tid == 0) {
        set_dev_status(a.dev_status, s_bad);
        a.accept_len[b] = 0;
        a.out_token[b] = -1;
      }
      for (int j = tid; j < N; j += blockDim.x) a.accepted[(size_t)b * N + j] = -1;
    }
    ptx::cluster_sync();
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
    const float l2p = s_l2p[u];
    const float l2q = s_l2q[u];
    // thread 0: raw logits of the next child's token, loaded while the rejection pass
    // before its decision runs (off the decision's critical path)
    float pre_x = 0.f, pre_y = 0.f;
    bool pre_ok = false;
    for (int k = 1; k <= m; ++k) {
      const int c = s_kids[k - 1];
      if (tid == 0) {
        const int t = s_tok[c];
        float pt, qt;
        if (res.nrej == 0) {
          pt = s_pc[c];
          qt = s_qc[c];
        } else {
          const float xt = pre_ok ? pre_x : ld_logit<T>(a.target, rowp + t);
          const float yt = pre_ok ? pre_y : ld_logit<T>(a.draft, rowp + t);
          const float p0 = ptx::ex2(fmaf(xt, a.c2, -l2p));
          const float q0 = ptx::ex2(fmaf(yt, a.c2, -l2q));
          eval_pq(res, t, p0, q0, pt, qt);
        }
        const float r = philox_uniform(a.seed, a.round, b, u, k, 0);
        const float alpha = qt > 0.f ? fminf(1.f, __fdiv_rn(pt, qt)) : (pt > 0.f ? 1.f : 0.f);
        s_dec = (r < alpha) ? 1 : 0;
        if (s_dec) s_found = c;
      }
      __syncthreads();
      if (s_dec) break;
      // loads thread 0 needs after the pass, issued before it: the rejected token's draft
      // logit and the next child's two logits
      float rej_y = 0.f;
      if (tid == 0) {
        rej_y = ld_logit<T>(a.draft, rowp + s_tok[c]);
        pre_ok = k < m;
        if (pre_ok) {
          const int tn = s_tok[s_kids[k]];
          pre_x = ld_logit<T>(a.target, rowp + tn);
          pre_y = ld_logit<T>(a.draft, rowp + tn);
        }
      }
      // rejection of t_k: Z = sum_v (P(v) - Q(v))+ with the current (P, Q)
      unsigned long long zs = 0;
      if (cached) {
        if (loaded_u != u || !loaded_q) load_rows(u, true);
        const float invd_n = res.invd[res.nrej];
        for (int i = tid; i < vhi - vlo; i += blockDim.x) {
          float P, q;
          cur_pq(i, P, q);
          zs += to_fix(fmaxf(P - q * invd_n, 0.f));
        }
        pend = false;
      } else
      for (int vb = vlo + tid; vb < vhi; vb += kBatch * blockDim.x) {
        float xs[kBatch], ys[kBatch];  // all loads of a batch in flight together
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int v = vb + i * blockDim.x;
          xs[i] = v < vhi ? ld_logit<T>(a.target, rowp + v) : 0.f;
          ys[i] = v < vhi ? ld_logit<T>(a.draft, rowp + v) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int v = vb + i * blockDim.x;
          if (v < vhi) {
            float P, Q;
            eval_pq(res, v, ptx::ex2(fmaf(xs[i], a.c2, -l2p)), ptx::ex2(fmaf(ys[i], a.c2, -l2q)), P, Q);
            zs += to_fix(fmaxf(P - Q, 0.f));
          }
        }
      }
      unsigned long long ztot = 0, dummy;
      block_scan_u64(zs, red, &ztot);
      const unsigned long long zall = cluster_total(ztot, &dummy);
      if (tid == 0) {
        const double z = (double)zall * 0x1p-56;
        const int j = res.nrej;
        const int t = s_tok[c];
        const float q0 = ptx::ex2(fmaf(rej_y, a.c2, -l2q));
        res.tok[j] = t;
        res.invz[j] = z > 0.0 ? (float)(1.0 / z) : 0.f;
        const float dprev = res.invd[j] > 0.f ? 1.f / res.invd[j] : 0.f;
        const float dnext = dprev - q0;
        res.invd[j + 1] = dnext > 0.f ? 1.f / dnext : 0.f;
        res.nrej = j + 1;
      }
      __syncthreads();
      if (cached) {
        // P_{n+1} = (P_n - Q_n)+ / Z_n where Z_n > 0 (else P stays), then t_k leaves Q:
        // applied element by element by the next sweep (each element is read and written
        // by the same thread)
        const int j = res.nrej - 1;
        pend = true;
        pend_invz = res.invz[j];
        pend_invd = res.invd[j];
        pend_tok = res.tok[j];
      }
    }
    if (s_found >= 0) {
      const int c = s_found;
      if (tid == 0 && crank == 0) a.accepted[(size_t)b * N + len] = c;
      ++len;
      u = c;
      __syncthreads();
      continue;
    }
    // ---- final draw from the current P by inverse CDF: smallest v with
    // target < prefix(v), target = floor(r * total), all in exact 2^-56 units
    const int per = (vhi - vlo + (int)blockDim.x - 1) / (int)blockDim.x;
    const int v0 = min(vhi, vlo + tid * per), v1 = min(vhi, v0 + per);
    // fixed-point terms P(v) of v0 + i, i < kBatch (below v1), loads issued together
    if (cached && loaded_u != u) load_rows(u, false);  // no rejection here: P = p
    if (cached && pend) {  // the last rejection's update, before P is read
      for (int i = tid; i < vhi - vlo; i += blockDim.x) {
        float P, q;
        cur_pq(i, P, q);
      }
      pend = false;
      __syncthreads();
    }
    auto terms = [&](int vb, unsigned long long* out) {
      if (cached) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int v = vb + i;
          out[i] = v < v1 ? to_fix(sP[v - vlo]) : 0ull;
        }
        return;
      }
      float xs[kBatch], ys[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int v = vb + i;
        xs[i] = v < v1 ? ld_logit<T>(a.target, rowp + v) : 0.f;
        ys[i] = (v < v1 && res.nrej) ? ld_logit<T>(a.draft, rowp + v) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int v = vb + i;
        out[i] = 0;
        if (v < v1) {
          float P, Q;
          eval_pq(res, v, ptx::ex2(fmaf(xs[i], a.c2, -l2p)), res.nrej ? ptx::ex2(fmaf(ys[i], a.c2, -l2q)) : 0.f,
                  P, Q);
          out[i] = to_fix(P);
        }
      }
    };
    unsigned long long loc = 0;
    for (int vb = v0; vb < v1; vb += kBatch) {
      unsigned long long tb[kBatch];
      terms(vb, tb);
#pragma unroll
      for (int i = 0; i < kBatch; ++i) loc += tb[i];
    }
    unsigned long long mine = 0, below = 0;
    const unsigned long long excl = block_scan_u64(loc, red, &mine);
    const unsigned long long total = cluster_total(mine, &below);
    const float r = philox_uniform(a.seed, a.round, b, u, 0, 1);
    const unsigned long long r24 = (unsigned long long)(r * 16777216.0f);  // r = k * 2^-24 exactly
    const unsigned long long target = (total >> 24) * r24 + (((total & 0xFFFFFFull) * r24) >> 24);
    if (total > 0) {
      const unsigned long long lo = below + excl;
      if (target >= lo && target < lo + loc) {
        // this thread's slice holds the crossing
        unsigned long long run = lo;
        int pick = v1 - 1;
        bool done = false;
        for (int vb = v0; vb < v1 && !done; vb += kBatch) {
          unsigned long long tb[kBatch];
          terms(vb, tb);
#pragma unroll
          for (int i = 0; i < kBatch; ++i) {
            run += tb[i];
            if (!done && vb + i < v1 && target < run) {
              pick = vb + i;
              done = true;
            }
          }
        }
        a.out_token[b] = pick;
      }
    } else if (tid == 0 && crank == 0) {
      a.out_token[b] = V - 1;
    }
    if (crank == 0) {
      if (tid == 0) a.accept_len[b] = len;
      for (int j = len + tid; j < N; j += blockDim.x) a.accepted[(size_t)b * N + j] = -1;
    }
    break;
  }
  ptx::cluster_sync();  // the other CTAs may still read this CTA's partial sums
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
  // 16 CTAs per cluster where the device can co-schedule them, else the portable 8
  // per device and element type (each kernel has its own attribute); 0 = not queried yet.
  // The release store follows the attribute change, so a thread that reads 16 launches
  // after the attribute is in place.
  static std::atomic<int> csize_cache[64][2];
  int dev = 0;
  cudaGetDevice(&dev);
  const int ti = dtype == TV_BF16 ? 1 : 0;
  int csize = (dev >= 0 && dev < 64) ? csize_cache[dev][ti].load(std::memory_order_acquire) : 0;
  if (csize == 0) {
    csize = 8;
    auto kern = dtype == TV_BF16 ? sample_walk_kernel<uint16_t> : sample_walk_kernel<float>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(kWalkClusterMax);
      q.blockDim = dim3(kWalkThreads);
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = kWalkClusterMax;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &q) == cudaSuccess && nclusters > 0)
        csize = kWalkClusterMax;
    }
    cudaGetLastError();  // a refused query leaves the portable size
    if (dev >= 0 && dev < 64) csize_cache[dev][ti].store(csize, std::memory_order_release);
  }
  a.csize = csize;
  const int span = (V + csize - 1) / csize;
  const size_t dyn = (size_t)((span + 3) & ~3) * 2 * sizeof(float);
  a.cached = dyn <= (size_t)kWalkDynCap ? 1 : 0;
  const size_t dsmem = a.cached ? dyn : 0;
  if (a.cached) {
    cudaError_t ea = dtype == TV_BF16
                         ? cudaFuncSetAttribute(sample_walk_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)dsmem)
                         : cudaFuncSetAttribute(sample_walk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)dsmem);
    if (ea != cudaSuccess) return ea;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B * csize);
  cfg.blockDim = dim3(kWalkThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaError_t e = dtype == TV_BF16
                      ? launch_pdl(sample_walk_kernel<uint16_t>, cfg.gridDim, cfg.blockDim, dsmem, stream, attr, 1, a)
                      : launch_pdl(sample_walk_kernel<float>, cfg.gridDim, cfg.blockDim, dsmem, stream, attr, 1, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tv
