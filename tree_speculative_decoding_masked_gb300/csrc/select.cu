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
#include "tv_ptx.cuh"

namespace tv {

constexpr int kSelThreads = 512;
constexpr int kSelCap = 4096;      // candidates held during the expansion
constexpr int kSelSlots = kSelCap + 32;  // + one spare slot per lane for masked-off stores
static_assert((size_t)kSelSlots * 28 + (size_t)kSelCap * 8 >= (size_t)kMaxBudget * 36,
              "the heap fallback fits below the pool copy");
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

// A second lower bound on the M-th best score, for large budgets, where the one-deviation
// family is sparse next to the whole candidate tree: count every candidate by its
// quantised log score.  (On a 16 x 4 pool at budget 64 it leaves 75 candidates instead
// of 238, but its 16 barrier-separated levels cost more than the expansion and ranking
// they save.)  Edge weight w = ceil(-16 log2 m + slack) >= -16 log2 m (16 bins
// per octave, 32 octaves; m = 0 or weights past the range are left out), so a path whose
// weights sum to <= v has an exact product >= 2^(-v/16); its fp32 product is within 16
// roundings of that, which the final scale covers.  H_l[v] = number of depth-l paths of
// weight v, built level by level (H_{l+1}[v] = sum over ranks of H_l[v - w]; counts
// saturate at 2^30).  The bound is 2^(-v*/16) (slightly shrunk) for the smallest v* whose
// paths of weight <= v* number at least M; 0 if the range holds fewer.
constexpr int kLogBins = kSelThreads;  // one weight bin per thread
constexpr int kCountMinRows = 128;     // smaller budgets use the one-deviation bound alone
constexpr unsigned kCountSat = 1u << 30;  // saturation of the per-bin path counts

__device__ float counting_bound(const SelSmem& sm, int d, int K, int M, unsigned long long* red, float* s_tau) {
  const int t = threadIdx.x;
  const int Kp = (K + 7) & ~7;                                            // ranks padded to whole groups of 8
  int* wts = sm.idx;                                  // [d][Kp] weights
  unsigned* H = reinterpret_cast<unsigned*>(sm.pos);  // [2][kLogBins] path counts, saturated
  for (int i = t; i < d * Kp; i += blockDim.x) {
    const int l = i / Kp, r = i - l * Kp;
    const float m = r < K ? sm.marg[l * K + r] : 0.f;
    int w = kLogBins;
    if (m > 0.f) {
      const float x = -16.f * log2f(m) + 1e-3f;
      if (x < (float)kLogBins) w = max((int)ceilf(x), 0);
    }
    wts[i] = w;
  }
  H[t] = t == 0 ? 1u : 0u;
  __syncthreads();
  unsigned long long acc = 0;
  for (int l = 0; l < d; ++l) {
    const unsigned* cur = H + (l & 1) * kLogBins;
    const int* wl = wts + l * Kp;
    unsigned long long h = 0;
    // weights grow with the rank: groups of 8 independent gathers until the first
    // weight past this thread's bin (no heavier edge can reach it)
    for (int r0 = 0; r0 < Kp && wl[r0] <= t; r0 += 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int w = wl[r0 + q];
        const unsigned x = cur[max(t - w, 0)];
        h += w <= t ? x : 0u;
      }
    }
    const unsigned hs = (unsigned)min(h, (unsigned long long)kCountSat);
    H[((l + 1) & 1) * kLogBins + t] = hs;
    acc += hs;
    __syncthreads();
  }
  unsigned long long tot;
  const unsigned long long excl = block_scan_u64(acc, red, &tot);
  if (t == 0) *s_tau = 0.f;
  __syncthreads();
  if (excl < (unsigned long long)M && excl + acc >= (unsigned long long)M)
    *s_tau = exp2f(-(float)t / 16.f) * (1.f - 1.f / 65536.f);
  __syncthreads();
  return *s_tau;
}

// Expand every candidate with s >= tau.  Each candidate lies on exactly one "run": a node
// reached by a rank >= 1 edge (or a child of the root), followed by its rank-0
// descendants.  Step 0 starts the runs at the root's children; step i+1 starts runs at
// the rank >= 1 children of every node made in step i.  One thread per (source node,
// rank) pair follows a run (its scores are a running fp32 product, exactly the
// left-to-right path product; the rank-0 factors m0 sit in registers); when the pairs
// outnumber the block, only the qualifying pairs are listed first (found per source by
// bisection over its sorted ranks).
// The number of steps is 1 + the largest number of rank >= 1 edges on a kept path.
// Step i counts its allocations in the set (i mod 3) of the counters: a set is cleared
// one step before its use and read by every thread one step after, so one barrier per
// step (two with the listing) orders everything.  Returns the entry count, or
// -(stored + 1) if more than kSelCap entries would be needed; then entries [0, stored)
// are complete (runs are allocated in increasing order, so the first run that did not
// fit ends the stored prefix) and prefix-closed.
struct ExpandCounters {
  int count[3];  // entries allocated by the step
  int fail[3];   // lowest offset that did not fit
  int live[3];   // (source, rank) pairs listed by the step
};

__device__ __forceinline__ int expand_threshold(const SelSmem& sm, const float (&m0)[kMaxDepth], int d, int K,
                                                float tau, ExpandCounters* ec) {
  const int t = threadIdx.x, lane = t & 31;
  if (t < 3) {
    ec->count[t] = 0;
    ec->fail[t] = 0x7fffffff;
    ec->live[t] = 0;
  }
  __syncthreads();
  int lo = 0, hi = 0;  // entries made by the previous step; step 0 expands the virtual root
  for (int step = 0, b = 0;; ++step, b = b == 2 ? 0 : b + 1) {
    const int nsrc = step == 0 ? 1 : hi - lo;
    const int r0 = step == 0 ? 0 : 1;
    const int nr = K - r0;
    if (nsrc <= 0 || nr <= 0) break;
    if (t == 0) {  // the set for step + 1 was last read before the previous barrier
      const int nb = b == 2 ? 0 : b + 1;
      ec->count[nb] = 0;
      ec->fail[nb] = 0x7fffffff;
      ec->live[nb] = 0;
    }
    int nitems = nsrc * nr;
    const float inv_nr = nr > 0 ? 1.f / (float)nr : 0.f;
    const bool listed = nitems > (int)blockDim.x;
    bool dropped = false;
    int* item = sm.pos;  // listed (source, rank) pairs, (entry + 1) << 8 | rank
    if (listed) {
      // per source the qualifying ranks form a prefix of [r0, K) (ranks are sorted and the
      // rounded product is monotone): count them by bisection, list every pair.  Each
      // pair makes at least one entry, so pairs past the free space are dropped and the
      // step then reports the overflow after storing what fits.
      for (int ib = t - lane; ib < nsrc; ib += blockDim.x) {
        const int i = ib + lane;
        int nq = 0, pe = -1;
        if (i < nsrc) {
          pe = step == 0 ? -1 : lo + i;
          const uint64_t pk0 = pe < 0 ? make_k0(1.f, 0) : sm.k0[pe];
          const int dep = (int)(pk0 & 0xFFFFFFFFu);
          if (dep < d) {
            const float ps = k0_score(pk0);
            const float* row = sm.marg + dep * K;
            int a = r0, z = K;  // the first rank in [r0, K] whose child misses tau
            while (a < z) {
              const int mid = (a + z) >> 1;
              if (__fmul_rn(ps, row[mid]) >= tau)
                a = mid + 1;
              else
                z = mid;
            }
            nq = a - r0;
          }
        }
        int incl = nq;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (total == 0) continue;
        int wb = 0;
        if (lane == 31) wb = atomicAdd(&ec->live[b], total);
        const int base = __shfl_sync(0xffffffffu, wb, 31) + incl - nq;
        for (int q = 0; q < nq && base + q < kSelCap - hi; ++q) item[base + q] = (pe + 1) << 8 | (r0 + q);
      }
      __syncthreads();
      nitems = ec->live[b];
      dropped = nitems > kSelCap - hi;
      if (dropped) nitems = kSelCap - hi;
    }
    // one thread per (source, rank): the run from that child
    for (int ib = t - lane; ib < nitems; ib += blockDim.x) {  // warp-uniform trip count
      const int it = ib + lane;
      int len = 0, pe = -1, dep = 0, r = 0;
      float s0 = 0.f;
      if (it < nitems) {
        if (listed) {
          const int v = item[it];
          pe = (v >> 8) - 1;
          r = v & 255;
        } else {
          int i = (int)((float)it * inv_nr);  // it / nr: the estimate is off by at most one
          if ((i + 1) * nr <= it)
            ++i;
          else if (i * nr > it)
            --i;
          r = r0 + (it - i * nr);
          pe = step == 0 ? -1 : lo + i;
        }
        const uint64_t pk0 = pe < 0 ? make_k0(1.f, 0) : sm.k0[pe];
        dep = (int)(pk0 & 0xFFFFFFFFu);  // children sit at position dep
        if (dep < d) {
          s0 = __fmul_rn(k0_score(pk0), sm.marg[dep * K + r]);
          // run length: the rank-r child, then rank-0 descendants while s >= tau.  The
          // products along a run never grow, so this is the count of its products that
          // reach tau; the multiply chain carries no compare.
          int cnt = 1;
          float sc = s0;
#pragma unroll
          for (int p = 1; p < kMaxDepth; ++p) {
            sc = __fmul_rn(sc, p > dep ? m0[p] : 1.f);
            cnt += (p > dep && p < d && sc >= tau) ? 1 : 0;
          }
          len = s0 >= tau ? cnt : 0;
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
      const int wmax = __reduce_max_sync(0xffffffffu, len);
      int wbase = 0;
      if (lane == 31) wbase = atomicAdd(&ec->count[b], total);
      const int base = hi + __shfl_sync(0xffffffffu, wbase, 31) + incl - len;
      if (len == 0) continue;
      if (base + len > kSelCap) {
        atomicMin(&ec->fail[b], base);
        continue;
      }
      uint64_t c1 = pe < 0 ? 0ull : sm.k1[pe], c2 = pe < 0 ? 0ull : sm.k2[pe];
      path_set(c1, c2, dep, r);
      // branch-free stores: entries outside the run go to the lane's spare slot.  Short
      // runs (every run of the warp within 4 or 8) walk 4 or 8 positions with the factors
      // read from shared memory up front; longer ones walk all positions with the factors
      // in registers.
      float sc = s0;
      if (wmax <= 8) {
        // the rank-0 factors of the next positions, loaded independently of each other;
        // 4 or 8 positions (warp-uniform)
        float f[8];
#pragma unroll
        for (int q = 1; q < 8; ++q) f[q] = sm.marg[min(dep + q, d - 1) * K];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (q == 4 && wmax <= 4) break;
          if (q > 0) sc = __fmul_rn(sc, f[q]);
          const int e = q < len ? base + q : kSelCap + lane;
          sm.k0[e] = make_k0(sc, dep + q + 1);
          sm.k1[e] = c1;
          sm.k2[e] = c2;
          sm.par[e] = q == 0 ? pe : e - 1;
        }
      } else {
#pragma unroll
        for (int p = 0; p < kMaxDepth; ++p) {
          const int q = p - dep;
          sc = __fmul_rn(sc, p > dep ? m0[p] : 1.f);
          const int e = (unsigned)q < (unsigned)len ? base + q : kSelCap + lane;
          sm.k0[e] = make_k0(sc, p + 1);
          sm.k1[e] = c1;
          sm.k2[e] = c2;
          sm.par[e] = q == 0 ? pe : e - 1;
        }
      }
    }
    __syncthreads();
    const int cnt = ec->count[b];
    int fail = ec->fail[b];
    if (dropped && fail == 0x7fffffff) fail = hi + cnt;  // everything allocated is stored
    if (fail != 0x7fffffff) {
      __syncthreads();  // every thread has read the set before a restart clears it
      return -fail - 1;
    }
    lo = hi;
    hi += cnt;
  }
  __syncthreads();  // every thread has read the last set before a restart clears it
  return hi;
}

constexpr int kFewChains = 128;  // up to this many chains share one histogram

// The one-deviation bound (see the top of this file): one coarse class histogram.
__device__ float family_bound(const SelSmem& sm, const float (&m0)[kMaxDepth], int d, int K, int M, int* hist,
                              int* bcast, float* s_tau) {
  const int t = threadIdx.x, lane = t & 31;
  // coarse histogram of the one-deviation candidates (ranks < kSelDevRanks).  Few
  // chains: spread over the warps (a few lanes each) into one shared histogram.  Many:
  // per-lane histogram columns (lane-major, in the expansion buffers, free for now), so
  // the atomics of a warp never collide.
  const int rmax = min(K, kSelDevRanks);
  const int nchain = 1 + d * (rmax - 1);  // chain 0: no deviation; else (position j, rank r)
  const bool few = nchain <= kFewChains;
  int* hcol = reinterpret_cast<int*>(sm.k1);
  if (few)
    hist[t] = 0;
  else
    for (int i = t; i < 32 * kSelBins / 4; i += blockDim.x) reinterpret_cast<int4*>(hcol)[i] = make_int4(0, 0, 0, 0);
  __syncthreads();
  int* mycol = few ? hist : hcol + lane * kSelBins;
  const int nw = blockDim.x >> 5;
  // few: chain c on lane c / nw of warp c % nw
  for (int c = few ? (lane * nw + (t >> 5)) : t; c < nchain; c += blockDim.x) {
    int j = -1, r = 0;
    if (c > 0) {
      j = (c - 1) / (rmax - 1);
      r = 1 + (c - 1) - j * (rmax - 1);
    }
    const float mj = j >= 0 ? sm.marg[j * K + r] : 1.f;
    float sc = 1.f;
    // the prefixes that contain the deviation are counted; the other positions add to
    // the lane's spare bin (branch-free)
#pragma unroll
    for (int p = 0; p < kMaxDepth; ++p) {
      sc = __fmul_rn(sc, p == j ? mj : m0[p]);
      atomicAdd(p < d && p >= j ? &mycol[score_class(sc)] : &hist[kSelBins + lane], 1);
    }
  }
  __syncthreads();
  if (!few) {
    int h = 0;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) h += hcol[l * kSelBins + t];
    hist[t] = h;
    __syncthreads();
  }
  return coarse_bound(hist, M, bcast + 2, s_tau);
}

constexpr int kRankDirect = 512;  // rank by direct comparison up to this many candidates

// Threshold selection by the block.  Returns 1 + number selected, or -1 if the
// candidate set did not fit (the caller falls back).
__device__ int select_threshold(const SelSmem& sm, int d, int K, int M, ExpandCounters* ec, int* s_count, int* hist,
                                int* bcast, float* s_tau, int32_t* o_par, int32_t* o_tok, int32_t* o_dep,
                                float* o_sc) {
  const int t = threadIdx.x;
  float m0[kMaxDepth];  // rank-0 factors, in registers for the run loops
#pragma unroll
  for (int p = 0; p < kMaxDepth; ++p) m0[p] = p < d ? sm.marg[p * K] : 1.f;
  // 1. a lower bound on the M-th best score: for small budgets the one-deviation bound
  // (cheap, and tight enough); for large ones the counting bound, which stays within a
  // few percent of M candidates where the one-deviation family is far too sparse
  float tau = M >= kCountMinRows ? counting_bound(sm, d, K, M, reinterpret_cast<unsigned long long*>(hist), s_tau)
                                 : 0.f;
  if (!(tau > 0.f)) tau = family_bound(sm, m0, d, K, M, hist, bcast, s_tau);
  // 2. expansion; restarts with tau raised to the M-th best stored score
  int n = -1;
  for (int attempt = 0; attempt <= kSelRetries; ++attempt) {
    n = expand_threshold(sm, m0, d, K, tau, ec);
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
    // With many more entries than places, rank only those at or above the coarse score
    // class where the count from the top reaches `take` (one histogram): at least `take`
    // entries lie above that class edge, so nothing below it is placed, and an entry's
    // rank among the listed ones is its rank among all.
    int nr = n;
    const int* list = nullptr;
    if (n > 2 * take && n > 64) {
      int* lst = reinterpret_cast<int*>(sm.k1 + (kSelCap - kRankDirect / 2));  // past every entry
      hist[t] = 0;
      if (t == 0) bcast[0] = 0;
      __syncthreads();
      if (t < n) atomicAdd(&hist[score_class(k0_score(sm.k0[t]))], 1);
      __syncthreads();
      const float edge = coarse_bound(hist, take, bcast + 2, s_tau);
      if (t < n && k0_score(sm.k0[t]) >= edge) lst[atomicAdd(&bcast[0], 1)] = t;
      __syncthreads();
      nr = bcast[0];
      list = lst;
    }
    // L lanes per entry (a power of two, L * nr <= blockDim): a branch-free count on the
    // (score, depth) word; exact ties are resolved on the rank path only when they occur
    int L = 1;
    while (L < 32 && 2 * L * nr <= (int)blockDim.x) L <<= 1;
    const int i_own = t / L, sub = t & (L - 1);
    const bool own = i_own < nr;
    const int e = own ? (list ? list[i_own] : i_own) : 0;
    const uint64_t a0 = own ? sm.k0[e] : 0ull;
    int less = 0, eq = 0;
    if (own) {
      int j = sub;
#pragma unroll 4
      for (; j < nr; j += L) {
        const uint64_t c = sm.k0[list ? list[j] : j];
        less += c < a0;
        eq += c == a0;
      }
    }
    for (int o = 1; o < L; o <<= 1) {
      less += __shfl_xor_sync(0xffffffffu, less, o);
      eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    int tied_before = 0;
    if (own && eq > 1) {
      const uint64_t a1 = sm.k1[e], a2 = sm.k2[e];
      for (int q0 = sub; q0 < nr; q0 += L) {
        const int q = list ? list[q0] : q0;
        if (sm.k0[q] == a0 && key_less(a0, sm.k1[q], sm.k2[q], a0, a1, a2)) ++tied_before;
      }
    }
    if (__any_sync(0xffffffffu, tied_before != 0))
      for (int o = 1; o < L; o <<= 1) tied_before += __shfl_xor_sync(0xffffffffu, tied_before, o);
    if (own && sub == 0) {
      const int rank = less + tied_before;
      sm.pos[e] = rank < take ? rank + 1 : 0;
      if (rank < take) sm.idx[rank] = e;
    }
  } else {
    // counting sort on the score bits: kSelCap bins over [tau, 1] (bin 0 = the highest
    // scores), then the exact order inside each bin by direct comparison
    static_assert(kSelCap % kSelThreads == 0, "whole bins per thread");
    constexpr int kPer = kSelCap / kSelThreads;
    int* cnt = sm.pos;   // bin counts, then bin ends
    int* list = sm.idx;  // entries grouped by bin
    const uint32_t u_hi = __float_as_uint(1.f), u_lo = __float_as_uint(tau);
    int shift = 0;
    while (((u_hi - u_lo) >> shift) >= (uint32_t)kSelCap) ++shift;
    auto bin_of = [&](uint64_t k0) {  // clamped, so out-of-range scores keep the order
      const uint32_t u = __float_as_uint(k0_score(k0));
      return u >= u_hi ? 0 : (int)((u_hi - max(u, u_lo)) >> shift);
    };
    for (int i = t; i < kSelCap; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    for (int e = t; e < n; e += blockDim.x) atomicAdd(&cnt[bin_of(sm.k0[e])], 1);
    __syncthreads();
    {  // exclusive scan: thread t owns bins [kPer t, kPer t + kPer)
      int c[kPer];
      unsigned long long own = 0;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        c[q] = cnt[kPer * t + q];
        own += c[q];
      }
      unsigned long long tot;
      int run = (int)block_scan_u64(own, reinterpret_cast<unsigned long long*>(hist), &tot);
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        cnt[kPer * t + q] = run;
        run += c[q];
      }
    }
    __syncthreads();
    for (int e = t; e < n; e += blockDim.x) list[atomicAdd(&cnt[bin_of(sm.k0[e])], 1)] = e;
    __syncthreads();  // cnt[b] is now the end of bin b
    int rk[kPer], en[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int j = t + q * kSelThreads;
      en[q] = -1;
      rk[q] = 0;
      if (j < n) {
        const int e = list[j];
        const uint64_t a0 = sm.k0[e], a1 = sm.k1[e], a2 = sm.k2[e];
        const int bn = bin_of(a0);
        const int lo = bn > 0 ? cnt[bn - 1] : 0, hi = cnt[bn];
        int rank = lo;
        for (int x = lo; x < hi; ++x) {
          const int f = list[x];
          const uint64_t c0 = sm.k0[f];
          rank += c0 < a0 || (c0 == a0 && key_less(c0, sm.k1[f], sm.k2[f], a0, a1, a2));
        }
        en[q] = e;
        rk[q] = rank;
      }
    }
    __syncthreads();  // the bins and the list are read; positions overwrite them
#pragma unroll
    for (int q = 0; q < kPer; ++q)
      if (en[q] >= 0) {
        sm.pos[en[q]] = rk[q] < take ? rk[q] + 1 : 0;
        if (rk[q] < take) sm.idx[rk[q]] = en[q];
      }
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
  __shared__ __align__(16) int hist[kSelBins + 32];  // + one spare bin per lane
  __shared__ int bcast[3 + kSelThreads / 32];
  __shared__ float s_tau;
  __shared__ int s_bad, s_nout, s_count;
  __shared__ ExpandCounters s_ec;
  const int b = blockIdx.x, tid = threadIdx.x;
  ptx::griddep_launch_dependents();  // the verification kernels may start their set-up
  ptx::griddep_wait();
  const int M = budget - 1;
  SelSmem sm;
  sm.k0 = reinterpret_cast<uint64_t*>(smem);
  sm.k1 = sm.k0 + kSelSlots;
  sm.k2 = sm.k1 + kSelSlots;
  sm.par = reinterpret_cast<int*>(sm.k2 + kSelSlots);
  sm.idx = sm.par + kSelSlots;
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
    const int r = select_threshold(sm, d, K, M, &s_ec, &s_count, hist, bcast, &s_tau, o_par, o_tok, o_dep, o_sc);
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
  const size_t expand = (size_t)kSelSlots * (3 * 8 + 4) + (size_t)kSelCap * 2 * 4;
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
  e = launch_pdl(select_kernel, dim3(B), dim3(kSelThreads), smem, stream, nullptr, 0, marg, ptok, d, K, budget,
                 root_token, parent, tokens, depth, score, n_nodes, dev_status, cost_base, cost_per_row);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tv
