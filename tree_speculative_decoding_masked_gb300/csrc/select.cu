// Budgeted prefix-closed subtree selection from a block-marginal pool.
//
// TAPS §4.1: d positions x top-K tokens form the candidate tree; §4.2: edge acceptance
// estimates propagate to path-level reach probabilities, and a prefix-closed subtree is
// kept greedily under the verification budget.  TreeGraft §3.1: cumulative path score
// s(v) = product of the edge scores along the root->v path, s(root) = 1.
// Edge score := the child's marginal; s is built with correctly rounded fp32 multiplies
// from the root down, so the result is reproducible bit for bit.
//
// Result: the first M = budget-1 candidates in the order (s desc, depth asc, rank path
// lexicographic asc), numbered in that order.  One CTA per sequence; the work is split
// into a few block-wide phases rather than budget-many serial steps:
//   1. a lower bound tau on the M-th best score, from the "one-deviation" candidates
//      (prefixes of the all-rank-0 path with at most one position replaced by a higher
//      rank): they are real candidates, so if at least M of them reach tau, so do at
//      least M candidates.  tau is the lower edge of the coarse score class (8 exponent
//      and 3 mantissa bits) in which their count from the top reaches M: one histogram.
//   2. expand the candidate tree keeping every node with s >= tau (scores never grow
//      along a path, so this set is prefix-closed and contains the answer), in parallel
//      over (node, rank) pairs.  If the set outgrows shared memory, tau is raised to the
//      M-th best score among the candidates already stored (again a valid bound) and the
//      expansion restarts;
//   3. order the set in the selection order (direct ranking when small, else an exact
//      cut at the M-th best score and a bitonic sort) and keep the first M.
// After a few failed restarts the kernel falls back to an exact best-first search by one
// warp (first-child / next-sibling form of the candidate tree, heap-ordered in the
// selection order).
#include "tv_kernels.cuh"

namespace tv {

constexpr int kSelThreads = 512;
constexpr int kSelCap = 4096;      // candidates held during the expansion
constexpr int kSelDevRanks = 32;   // ranks 1..31 enumerated in the one-deviation family
constexpr int kSelBins = 512;      // coarse score classes of [2^-63, 1]: 8 per octave, the lowest takes the rest
constexpr int kSelRetries = 4;     // expansions with a raised bound before the fallback
static_assert(kSelBins == kSelThreads, "one coarse class per thread");
static_assert(32 * kSelBins * 4 <= 2 * kSelCap * 8, "per-lane histogram columns fit in two key arrays");

__device__ __forceinline__ bool key_less(uint64_t a0, uint64_t a1, uint64_t a2, uint64_t b0, uint64_t b1,
                                         uint64_t b2) {
  if (a0 != b0) return a0 < b0;
  if (a1 != b1) return a1 < b1;
  return a2 < b2;
}

// Rank path packed one byte per level, level 0 in the top byte of k1, level 8 in k2.
__device__ __forceinline__ int path_rank(uint64_t k1, uint64_t k2, int level) {
  return level < 8 ? (int)((k1 >> (8 * (7 - level))) & 0xFF) : (int)((k2 >> (8 * (15 - level))) & 0xFF);
}
__device__ __forceinline__ void path_set(uint64_t& k1, uint64_t& k2, int level, int r) {
  if (level < 8)
    k1 |= (uint64_t)r << (8 * (7 - level));
  else
    k2 |= (uint64_t)r << (8 * (15 - level));
}
__device__ __forceinline__ void path_bump(uint64_t& k1, uint64_t& k2, int level) {
  if (level < 8)
    k1 += 1ull << (8 * (7 - level));
  else
    k2 += 1ull << (8 * (15 - level));
}
// k0 = (~bits(s)) << 32 | depth: larger s (s >= 0) gives a smaller key
__device__ __forceinline__ uint64_t make_k0(float s, int depth) {
  return ((uint64_t)(~__float_as_uint(s)) << 32) | (uint32_t)depth;
}
__device__ __forceinline__ float k0_score(uint64_t k0) { return __uint_as_float(~(uint32_t)(k0 >> 32)); }

// ------------------------------------------------------------------------------------
// exact best-first search by one warp (fallback)

__device__ int select_heap_warp(const float* sm_marg, const int* sm_tok, int d, int K, int budget,
                                unsigned char* work, int32_t* o_par, int32_t* o_tok, int32_t* o_dep, float* o_sc) {
  const int lane = threadIdx.x & 31;
  const int cap = budget;  // frontier never exceeds 1 + pops <= budget
  uint64_t* k0 = reinterpret_cast<uint64_t*>(work);
  uint64_t* k1 = k0 + cap;
  uint64_t* k2 = k1 + cap;
  int* par = reinterpret_cast<int*>(k2 + cap);
  float* psc = reinterpret_cast<float*>(par + cap);
  int F = 0;
  if (d >= 1 && K >= 1 && budget > 1) {
    if (lane == 0) {
      k0[0] = make_k0(__fmul_rn(1.f, sm_marg[0]), 1);
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
      const float s = k0_score(b0);
      const int p = par[bi];
      const float ps = psc[bi];
      const int r = path_rank(b1, b2, dep - 1);
      o_par[n] = p;
      o_tok[n] = sm_tok[(dep - 1) * K + r];
      o_dep[n] = dep;
      o_sc[n] = s;
      const int last = F - 1;
      k0[bi] = k0[last];
      k1[bi] = k1[last];
      k2[bi] = k2[last];
      par[bi] = par[last];
      psc[bi] = psc[last];
      int f = last;
      if (dep < d) {  // first child: rank 0 at the next position
        k0[f] = make_k0(__fmul_rn(s, sm_marg[dep * K]), dep + 1);
        k1[f] = b1;
        k2[f] = b2;
        par[f] = n;
        psc[f] = s;
        ++f;
      }
      if (r + 1 < K) {  // next sibling under the same parent
        uint64_t n1 = b1, n2 = b2;
        path_bump(n1, n2, dep - 1);
        k0[f] = make_k0(__fmul_rn(ps, sm_marg[(dep - 1) * K + r + 1]), dep);
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
  return n;
}

// ------------------------------------------------------------------------------------
// block helpers (kSelThreads threads)

// Radix select of the k-th largest (1-based, k <= n) of vals[0..n) with warp-aggregated
// histogram updates.  With min_shift = 0 the exact value is returned; with a larger
// min_shift the passes stop early and the result is the k-th largest value with its low
// min_shift bits cleared (a lower bound).  Every thread returns the result.
__device__ uint32_t block_kth_largest(const uint32_t* vals, int n, int k, int* hist, int* bcast, int min_shift = 0) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, mask = 0;
  int want = k;
  for (int shift = 24; shift >= min_shift; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const uint32_t v = i < n ? vals[i] : 0u;
      const bool act = i < n && (v & mask) == prefix;
      const unsigned am = __ballot_sync(0xffffffffu, act);
      if (act) {
        const int dig = (int)((v >> shift) & 255u);
        const unsigned peers = __match_any_sync(am, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[dig], __popc(peers));
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int cnt[8];
      int tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // lane l owns digits 255-8l .. 248-8l
        cnt[j] = hist[255 - 8 * lane - j];
        tot += cnt[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < want && incl >= want);
      const int src = hit ? __ffs(hit) - 1 : 0;
      if (lane == src) {
        int dig = 0, rest = 1;
        if (hit) {
          int run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run + cnt[j] >= want) {
              dig = 255 - 8 * lane - j;
              rest = want - run;
              break;
            }
            run += cnt[j];
          }
        }
        bcast[0] = dig;
        bcast[1] = rest;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)bcast[0] << shift;
    mask |= 255u << shift;
    want = bcast[1];
    __syncthreads();
  }
  return prefix;
}

struct SelSmem {
  float* marg;
  int* tok;
  uint64_t* k0;
  uint64_t* k1;
  uint64_t* k2;
  int* par;   // parent entry (-1: the root)
  int* idx;   // sort permutation
  int* pos;   // entry -> position in the output (0: not taken)
};

// Coarse score class of s in [0, 1]: 8 exponent and 3 mantissa bits (8 classes per
// octave), offset so that class 1 starts at 2^-63; class 0 holds everything below.
__device__ __forceinline__ int score_class(float s) {
  return min(max((int)(__float_as_uint(s) >> 20) - 512, 0), kSelBins - 1);
}
__device__ __forceinline__ float class_floor(int c) { return c <= 0 ? 0.f : __uint_as_float((uint32_t)(c + 512) << 20); }

// Lower edge of the highest class c such that the histogram's count in classes >= c
// reaches M; 0 if the total is below M.  One class per thread (kSelBins == blockDim.x).
__device__ float coarse_bound(const int* hist, int M, int* wsum, float* s_tau) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int c = kSelBins - 1 - t;  // this thread's class, in descending score order
  const int h = hist[c];
  int incl = h;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[w] = incl;
  if (t == 0) *s_tau = 0.f;
  __syncthreads();
  int before = 0;
  for (int k = 0; k < w; ++k) before += wsum[k];
  const int excl = before + incl - h;
  if (excl < M && excl + h >= M) *s_tau = class_floor(c);
  __syncthreads();
  return *s_tau;
}

// Expand every candidate with s >= tau.  Each candidate lies on exactly one "run": a node
// reached by a rank >= 1 edge (or a child of the root), followed by its rank-0
// descendants.  Step 0 starts the runs at the root's children; step i+1 starts runs at
// the rank >= 1 children of every node made in step i.  Per step, the nodes with at
// least one qualifying child are listed first; then one thread per (listed node, rank)
// pair follows a run (its scores are a running fp32 product, exactly the left-to-right
// path product).  The number of steps is 1 + the largest number of rank >= 1 edges on a
// kept path.  Returns the entry count, or -(stored + 1) if more than kSelCap entries would
// be needed; then entries [0, stored) are complete (runs are allocated in increasing
// order, so the first run that did not fit ends the stored prefix) and prefix-closed.
__device__ __forceinline__ int expand_threshold(const SelSmem& sm, int d, int K, float tau, int* s_count,
                                                int* s_fail, int* s_live) {
  const int t = threadIdx.x, lane = t & 31;
  int* live = sm.idx;  // sources with a qualifying child, this step
  if (t == 0) {
    *s_count = 0;
    *s_fail = 0x7fffffff;
    *s_live = 0;
  }
  __syncthreads();
  int lo = 0, hi = 0;  // entries made by the previous step; step 0 expands the virtual root
  for (int step = 0;; ++step) {
    const int nsrc = step == 0 ? 1 : hi - lo;
    if (nsrc <= 0) break;
    const int r0 = step == 0 ? 0 : 1;
    const int nr = K - r0;
    if (nr <= 0) break;
    // 1. sources whose best rank >= r0 child reaches tau (ranks are sorted)
    for (int ib = t - lane; ib < nsrc; ib += blockDim.x) {
      const int i = ib + lane;
      bool ok = false;
      if (i < nsrc) {
        const uint64_t pk0 = step == 0 ? make_k0(1.f, 0) : sm.k0[lo + i];
        const int dep = (int)(pk0 & 0xFFFFFFFFu);
        ok = dep < d && __fmul_rn(k0_score(pk0), sm.marg[dep * K + r0]) >= tau;
      }
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (m == 0) continue;
      int wb = 0;
      if (lane == 0) wb = atomicAdd(s_live, __popc(m));
      wb = __shfl_sync(0xffffffffu, wb, 0);
      if (ok) live[wb + __popc(m & ((1u << lane) - 1))] = step == 0 ? -1 : lo + i;
    }
    __syncthreads();
    const int nlive = *s_live;
    __syncthreads();
    if (t == 0) *s_live = 0;
    // 2. one thread per (listed source, rank): the run from that child
    const int items = nlive * nr;
    for (int ib = t - lane; ib < items; ib += blockDim.x) {  // warp-uniform trip count
      const int it = ib + lane;
      int len = 0, pe = -1, dep = 0, r = 0;
      float s0 = 0.f;
      if (it < items) {
        const int i = it / nr;
        r = r0 + (it - i * nr);
        pe = live[i];
        const uint64_t pk0 = pe < 0 ? make_k0(1.f, 0) : sm.k0[pe];
        dep = (int)(pk0 & 0xFFFFFFFFu);  // children sit at position dep
        s0 = __fmul_rn(k0_score(pk0), sm.marg[dep * K + r]);
        if (s0 >= tau) {
          // run length: the rank-r child, then rank-0 descendants while s >= tau
          len = 1;
          float sc = s0;
          for (int p = dep + 1; p < d; ++p) {
            const float nx = __fmul_rn(sc, sm.marg[p * K]);
            if (!(nx >= tau)) break;
            sc = nx;
            ++len;
          }
        }
      }
      // one allocation per warp: lanes take consecutive slots in lane order
      int incl = len;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (total == 0) continue;
      int wbase = 0;
      if (lane == 31) wbase = atomicAdd(s_count, total);
      const int base = __shfl_sync(0xffffffffu, wbase, 31) + incl - len;
      if (len == 0) continue;
      if (base + len > kSelCap) {
        atomicMin(s_fail, base);
        continue;
      }
      uint64_t c1 = pe < 0 ? 0ull : sm.k1[pe], c2 = pe < 0 ? 0ull : sm.k2[pe];
      path_set(c1, c2, dep, r);
      float sc = s0;
      for (int q = 0; q < len; ++q) {
        if (q > 0) sc = __fmul_rn(sc, sm.marg[(dep + q) * K]);
        const int e = base + q;
        sm.k0[e] = make_k0(sc, dep + q + 1);
        sm.k1[e] = c1;
        sm.k2[e] = c2;
        sm.par[e] = q == 0 ? pe : e - 1;
      }
    }
    __syncthreads();
    const int fail = *s_fail, cnt = *s_count;
    __syncthreads();  // every thread has read the counters before the next step moves them
    if (fail != 0x7fffffff) return -fail - 1;
    lo = hi;
    hi = cnt;
  }
  return hi;
}

// bitonic sort of sm.idx[0..n2) (entries, -1 = padding last) in the selection order
__device__ void bitonic_sort_idx(const SelSmem& sm, int n2) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n2 / 2; i += blockDim.x) {
        const int lo = 2 * stride * (i / stride) + (i % stride);
        const int hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const int a = sm.idx[lo], c = sm.idx[hi];
        bool a_gt;
        if (a < 0)
          a_gt = c >= 0;
        else if (c < 0)
          a_gt = false;
        else
          a_gt = key_less(sm.k0[c], sm.k1[c], sm.k2[c], sm.k0[a], sm.k1[a], sm.k2[a]);
        if (a_gt == asc) {
          sm.idx[lo] = c;
          sm.idx[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

constexpr int kRankDirect = 512;  // rank by direct comparison up to this many candidates

// Threshold selection by the block.  Returns 1 + number selected, or -1 if the
// candidate set did not fit (the caller falls back).
__device__ int select_threshold(const SelSmem& sm, int d, int K, int M, int* s_count, int* s_fail, int* hist,
                                int* bcast, float* s_tau, int32_t* o_par, int32_t* o_tok, int32_t* o_dep,
                                float* o_sc) {
  const int t = threadIdx.x;
  // 1. coarse histogram of the one-deviation candidates (ranks < kSelDevRanks)
  // per-lane histogram columns (lane-major, in the expansion buffers, free for now): the
  // atomics of a warp never collide
  int* hcol = reinterpret_cast<int*>(sm.k1);
  for (int i = t; i < 32 * kSelBins / 4; i += blockDim.x) reinterpret_cast<int4*>(hcol)[i] = make_int4(0, 0, 0, 0);
  float m0[kMaxDepth];  // rank-0 factors, in registers for the run loops
#pragma unroll
  for (int p = 0; p < kMaxDepth; ++p) m0[p] = p < d ? sm.marg[p * K] : 1.f;
  __syncthreads();
  const int rmax = min(K, kSelDevRanks);
  const int nchain = 1 + d * (rmax - 1);  // chain 0: no deviation; else (position j, rank r)
  const int lane = t & 31;
  int* mycol = hcol + lane * kSelBins;
  for (int c = t; c < nchain; c += blockDim.x) {
    int j = -1, r = 0;
    if (c > 0) {
      j = (c - 1) / (rmax - 1);
      r = 1 + (c - 1) - j * (rmax - 1);
    }
    const float mj = j >= 0 ? sm.marg[j * K + r] : 1.f;
    float sc = 1.f;
#pragma unroll
    for (int p = 0; p < kMaxDepth; ++p) {
      if (p < d) {
        sc = __fmul_rn(sc, p == j ? mj : m0[p]);
        if (p >= j) atomicAdd(&mycol[score_class(sc)], 1);  // prefixes that contain the deviation
      }
    }
  }
  __syncthreads();
  {
    int h = 0;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) h += hcol[l * kSelBins + t];
    hist[t] = h;
  }
  __syncthreads();
  float tau = coarse_bound(hist, M, bcast + 2, s_tau);
  // 2. expansion; restarts with tau raised to the M-th best stored score
  int n = -1;
  for (int attempt = 0; attempt <= kSelRetries; ++attempt) {
    n = expand_threshold(sm, d, K, tau, s_count, s_fail, bcast + 2 + kSelThreads / 32);
    if (n >= 0) break;
    const int stored = -n - 1;
    n = -1;
    if (stored < M || attempt == kSelRetries) break;
    uint32_t* sc = reinterpret_cast<uint32_t*>(sm.idx);
    for (int i = t; i < stored; i += blockDim.x) sc[i] = __float_as_uint(k0_score(sm.k0[i]));
    __syncthreads();
    const float raised = __uint_as_float(block_kth_largest(sc, stored, M, hist, bcast));
    __syncthreads();
    if (!(raised > tau)) break;  // ties at the bound: no progress possible
    tau = raised;
  }
  if (n < 0) return -1;
  const int take = min(n, M);
  // 3. order: the output position of entry e is 1 + its rank in the selection order
  if (n <= kRankDirect) {
    for (int e = t; e < n; e += blockDim.x) {
      // branch-free count on the (score, depth) word; exact ties are resolved on the
      // rank path only when they occur
      const uint64_t a0 = sm.k0[e];
      int less = 0, eq = 0;
      int j = 0;
      const ulonglong2* k0v = reinterpret_cast<const ulonglong2*>(sm.k0);
#pragma unroll 4
      for (; j + 2 <= n; j += 2) {
        const ulonglong2 c = k0v[j >> 1];
        less += (c.x < a0) + (c.y < a0);
        eq += (c.x == a0) + (c.y == a0);
      }
      if (j < n) {
        less += sm.k0[j] < a0;
        eq += sm.k0[j] == a0;
      }
      int rank = less;
      if (eq > 1) {
        const uint64_t a1 = sm.k1[e], a2 = sm.k2[e];
        for (int q = 0; q < n; ++q)
          if (sm.k0[q] == a0 && key_less(a0, sm.k1[q], sm.k2[q], a0, a1, a2)) ++rank;
      }
      sm.pos[e] = rank < take ? rank + 1 : 0;
      if (rank < take) sm.idx[rank] = e;
    }
  } else {
    // only entries with s >= (M-th best score) can be taken: sort just those
    uint32_t* sc = reinterpret_cast<uint32_t*>(sm.pos);
    for (int i = t; i < n; i += blockDim.x) sc[i] = __float_as_uint(k0_score(sm.k0[i]));
    __syncthreads();
    const uint32_t T = block_kth_largest(sc, n, take, hist, bcast);
    if (t == 0) *s_count = 0;
    __syncthreads();
    for (int i = t; i < n; i += blockDim.x)
      if (sc[i] >= T) sm.idx[atomicAdd(s_count, 1)] = i;
    __syncthreads();
    const int cnt_ge = *s_count;
    int n2 = 1;
    while (n2 < cnt_ge) n2 <<= 1;
    if (n2 > 2 * kSelCap) return -1;
    for (int i = cnt_ge + t; i < n2; i += blockDim.x) sm.idx[i] = -1;
    __syncthreads();
    bitonic_sort_idx(sm, n2);
    for (int i = t; i < take; i += blockDim.x) sm.pos[sm.idx[i]] = i + 1;
  }
  __syncthreads();
  for (int i = t; i < take; i += blockDim.x) {
    const int e = sm.idx[i];
    const uint64_t k0 = sm.k0[e];
    const int dep = (int)(k0 & 0xFFFFFFFFu);
    const int r = path_rank(sm.k1[e], sm.k2[e], dep - 1);
    o_par[i + 1] = sm.par[e] < 0 ? 0 : sm.pos[sm.par[e]];
    o_tok[i + 1] = sm.tok[(dep - 1) * K + r];
    o_dep[i + 1] = dep;
    o_sc[i + 1] = k0_score(k0);
  }
  __syncthreads();
  return 1 + take;
}

// TAPS §3.1 (limitation 2) and §3.2: verify the prefix of the selection order that
// maximises expected tokens per unit of verification cost.  Expected tokens of the first
// n rows = 1 + sum of the drafts' s (each s(v) is v's acceptance probability under the
// edge-score reading, plus the round's bonus token); cost = cost_base + cost_per_row * n.
// Scores are rounded to multiples of 2^-40 and summed exactly (64-bit integers), the
// ratio is one IEEE double division; n* is the smallest maximiser.  Needs the CTA's
// output writes to be complete (called after a barrier).
constexpr float kFixUnit = 1099511627776.0f;  // 2^40

__device__ int cost_aware_rows(const float* o_sc, int n_out, float cost_base, float cost_per_row) {
  __shared__ unsigned long long red[33];
  __shared__ double s_obj[32];
  __shared__ int s_n[32];
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int T = blockDim.x;
  __syncthreads();
  // rows 1 .. n_out-1 in contiguous slices
  const int nd = n_out - 1;
  const int per = (nd + T - 1) / T;
  const int r0 = 1 + t * per, r1 = min(n_out, r0 + per);
  unsigned long long loc = 0;
  for (int r = r0; r < r1; ++r) loc += __float2ull_rn(o_sc[r] * kFixUnit);
  unsigned long long tot;
  unsigned long long acc = block_scan_u64(loc, red, &tot);
  const double a = (double)cost_base, bcost = (double)cost_per_row;
  auto objective = [&](unsigned long long sum, int n) {
    const double num = (double)(1099511627776ull + sum);
    return __ddiv_rn(num, __dadd_rn(a, __dmul_rn(bcost, (double)n)));
  };
  double best = t == 0 ? objective(0ull, 1) : -1.0;
  int best_n = t == 0 ? 1 : 0x7fffffff;
  for (int r = r0; r < r1; ++r) {
    acc += __float2ull_rn(o_sc[r] * kFixUnit);
    const double v = objective(acc, r + 1);
    if (v > best) {  // rows grow within the slice: a later row wins only if strictly better
      best = v;
      best_n = r + 1;
    }
  }
  // largest objective, smallest n among equals
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int on = __shfl_xor_sync(0xffffffffu, best_n, o);
    if (ov > best || (ov == best && on < best_n)) {
      best = ov;
      best_n = on;
    }
  }
  if (lane == 0) {
    s_obj[wid] = best;
    s_n[wid] = best_n;
  }
  __syncthreads();
  if (wid == 0) {
    best = lane < (T >> 5) ? s_obj[lane] : -1.0;
    best_n = lane < (T >> 5) ? s_n[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int on = __shfl_xor_sync(0xffffffffu, best_n, o);
      if (ov > best || (ov == best && on < best_n)) {
        best = ov;
        best_n = on;
      }
    }
    if (lane == 0) s_n[0] = best_n;
  }
  __syncthreads();
  const int n = s_n[0];
  __syncthreads();
  return n;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float* __restrict__ marg,
                                                             const int32_t* __restrict__ ptok, int d, int K,
                                                             int budget, const int32_t* __restrict__ root_token,
                                                             int32_t* out_parent, int32_t* out_tok, int32_t* out_depth,
                                                             float* out_score, int32_t* n_nodes, int32_t* dev_status,
                                                             float cost_base, float cost_per_row) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int hist[kSelBins > 256 ? kSelBins : 256];
  __shared__ int bcast[3 + kSelThreads / 32];
  __shared__ float s_tau;
  __shared__ int s_bad, s_nout, s_count, s_fail;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int M = budget - 1;
  SelSmem sm;
  sm.k0 = reinterpret_cast<uint64_t*>(smem);
  sm.k1 = sm.k0 + kSelCap;
  sm.k2 = sm.k1 + kSelCap;
  sm.par = reinterpret_cast<int*>(sm.k2 + kSelCap);
  sm.idx = sm.par + kSelCap;
  sm.pos = sm.idx + kSelCap;
  sm.marg = reinterpret_cast<float*>(sm.pos + kSelCap);
  sm.tok = reinterpret_cast<int*>(sm.marg + d * K);

  const float* mg = marg + (size_t)b * d * K;
  const int32_t* tk = ptok + (size_t)b * d * K;
  const int root = (tid == 0 && root_token) ? root_token[b] : -1;  // in flight with the pool loads
  if (tid == 0) {
    s_bad = 0;
    s_nout = -1;
  }
  __syncthreads();
  for (int i = tid; i < d * K; i += blockDim.x) {
    const float m = mg[i];
    sm.marg[i] = m;
    sm.tok[i] = tk[i];
    const bool sorted = (i % K == 0) || !(m > mg[i - 1]);
    if (!(m >= 0.f && m <= 1.f) || !sorted) s_bad = 1;
  }
  __syncthreads();
  if (s_bad && tid == 0) set_dev_status(dev_status, TV_DEV_BAD_TOKEN);

  int32_t* o_par = out_parent + (size_t)b * budget;
  int32_t* o_tok = out_tok + (size_t)b * budget;
  int32_t* o_dep = out_depth + (size_t)b * budget;
  float* o_sc = out_score + (size_t)b * budget;
  if (tid == 0) {
    o_par[0] = -1;
    o_tok[0] = root;
    o_dep[0] = 0;
    o_sc[0] = 1.f;
  }
  if (M <= 0) {
    if (tid == 0) s_nout = 1;
  } else if (M <= kSelCap / 2) {
    const int r = select_threshold(sm, d, K, M, &s_count, &s_fail, hist, bcast, &s_tau, o_par, o_tok, o_dep, o_sc);
    if (tid == 0) s_nout = r;
  }
  __syncthreads();
  if (s_nout < 0) {
    // exact fallback: best-first search by warp 0 over the whole shared buffer
    if (tid < 32) {
      const int r = select_heap_warp(sm.marg, sm.tok, d, K, budget, smem, o_par, o_tok, o_dep, o_sc);
      if (tid == 0) s_nout = r;
    }
    __syncthreads();
  }
  int n_out = s_nout;
  if (cost_per_row > 0.f && n_out > 1) n_out = cost_aware_rows(o_sc, n_out, cost_base, cost_per_row);
  for (int j = n_out + tid; j < budget; j += blockDim.x) {
    o_par[j] = -1;
    o_tok[j] = -1;
    o_dep[j] = -1;
    o_sc[j] = 0.f;
  }
  if (tid == 0 && n_nodes) n_nodes[b] = n_out;
}

static size_t select_smem_bytes(int d, int K, int budget) {
  const size_t expand = (size_t)kSelCap * (3 * 8 + 3 * 4);
  const size_t heap = (size_t)budget * (3 * 8 + 4 + 4);
  // the heap fallback reuses the start of the buffer; marg/tok follow the expansion arrays
  return (expand > heap ? expand : heap) + (size_t)d * K * 8;
}

size_t select_ws_bytes(int, int, int, int) { return 0; }

cudaError_t launch_select(const float* marg, const int32_t* ptok, int B, int d, int K, int budget,
                          const int32_t* root_token, int32_t* parent, int32_t* tokens, int32_t* depth,
                          float* score, int32_t* n_nodes, char*, int32_t* dev_status, float cost_base,
                          float cost_per_row, cudaStream_t stream) {
  const size_t smem = select_smem_bytes(d, K, budget);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  select_kernel<<<B, kSelThreads, smem, stream>>>(marg, ptok, d, K, budget, root_token, parent, tokens, depth, score,
                                                   n_nodes, dev_status, cost_base, cost_per_row);
  return cudaGetLastError();
}

}  // namespace tv
