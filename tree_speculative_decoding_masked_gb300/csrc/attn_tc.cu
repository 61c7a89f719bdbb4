// Tree-masked GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// PTD §3.1: node i attends to the committed prefix and to its observable set pi(i);
// TAPS §4.1: the selected subtree is verified by the target in one pass with tree
// attention.  Three kernels share this file: attn_tc_kernel (one 128-row tile per CTA,
// described here), attn_pair_kernel (two row tiles per CTA) and attn_pair2_kernel (two
// row tiles, 64-key KV tiles, two S buffers per row tile), each described where it is
// defined; the host side at the end picks one per launch from a wave model.
// attn_tc_kernel: one CTA owns a tile of 128 query rows that share one KV head: the G query
// heads of a GQA group times NT = 128/G consecutive tree nodes (head-major rows), so each
// K/V tile fetched from HBM by TMA is used by every node and every head of the group.
// The key range [0, P + last node of the tile) is cut into KV splits across CTAs.
//
// Per CTA, warp-specialised:
//   warp 0      TMA producers: lane 0 loads the Q tile once, then K tiles of 128 keys
//               into a 3-slot ring; lane 1 loads the V tiles into a 2-slot ring
//   warp 1      TMEM owner; lane 0 issues S[t&1] = Q K_t^T (M=128, N=128, K=D, fp32
//               in TMEM) as soon as a K tile and an S buffer are free
//   warp 10     lane 0 issues O += P_t V_t (M=128, N=D, K=128, fp32 in TMEM, P_t read
//               from TMEM) as soon as the softmax has written P_t
//   warps 2..9  softmax: two threads per row (each half of a tile's 128 keys); read S
//               from TMEM, apply the tree mask, agree on the row max with the partner
//               thread, keep a running reference max (rescale O only when the max grows
//               by more than 2^8), write P (bf16) into one of two TMEM buffers, so the
//               exponentials of tile t overlap the PV product of tile t-1.
// TMEM columns: S[0] 0..127, S[1] 128..255, O 256..256+D, P[0] 384..447, P[1] 448..511.
// With one split the epilogue normalises O and stores bf16.  With several, the splits of
// a row tile run as one thread-block cluster: each CTA parks its unnormalised O and
// (m, l) in its own shared memory and, after a cluster barrier, merges a slice of the
// rows by reading its peers' partials over distributed shared memory.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "tv_kernels.cuh"
#include "tv_ptx.cuh"

namespace tv {

constexpr int kRows = 128;     // MMA M: query rows per CTA
constexpr int kBN = 128;       // keys per KV tile (MMA N of QK^T, K of PV)
constexpr int kKSlots = 3;     // K ring depth (tiles of 128 keys)
constexpr int kVSlots = 2;     // V ring depth
constexpr int kThreads = 352;  // 11 warps: TMA producers, S issuer, 8 softmax warps, PV issuer
constexpr float kRescaleLog2 = 8.f;
constexpr float kRescaleSum = 256.f;  // 2^kRescaleLog2
constexpr int kMaxSplits = 8;  // KV splits of a row tile = one portable-size cluster

template <int D>
struct TcCfg {
  static constexpr int kDB = D / 64;                  // 64-element (128-byte) column blocks
  static constexpr int kQBlock = kRows * 128;         // bytes per column block of Q
  static constexpr int kKVBlock = kBN * 128;          // bytes per column block of a K or V tile
  static constexpr int kQBytes = kDB * kQBlock;
  static constexpr int kTileBytes = kDB * kKVBlock;   // one K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKSlots * kTileBytes;
  static constexpr int kOffPar = kOffV + kVSlots * kTileBytes;
  static constexpr int kOffBar = kOffPar + kMaxNodes * 4;
  static constexpr int kSmemUsed = kOffBar + 256;
  static constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 2 * kBN;           // after S[0], S[1]
  static constexpr uint32_t kColP = 384;               // P[0], P[1]: 64 columns each
  static_assert(kColO + D <= kColP && kColP + 2 * (kBN / 2) <= kTmemCols, "TMEM budget");
  static_assert(kOffV - kOffK >= D * kRows * 4 + kRows * 8, "split partials fit in the drained K ring");
};

struct TcArgs {
  void* out;
  const int32_t* parent;
  int B, Hq, Hkv, N, P, G, NT, MT, splits;
  int mcast;  // attn_pair2_kernel: tile pairs 2c and 2c + 1 form a cluster sharing each K/V tile
  float c;  // softmax scale * log2(e)
  int32_t* dev_status;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKSlots];
  uint64_t k_empty[kKSlots];
  uint64_t v_full[kVSlots];
  uint64_t v_empty[kVSlots];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];  // PV(t) complete, on barrier t & 1
  uint64_t o_done;
  uint64_t s_done;
  uint32_t tmem_base;
  int abort;
};

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// max of `init` and 64 scores: four independent chains of three-input maxima
__device__ __forceinline__ float max64(const float (&sv)[64], float init) {
  float c0 = init, c1 = -INFINITY, c2 = -INFINITY, c3 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; j += 8) {
    c0 = fmax3(c0, sv[j], sv[j + 1]);
    c1 = fmax3(c1, sv[j + 2], sv[j + 3]);
    c2 = fmax3(c2, sv[j + 4], sv[j + 5]);
    c3 = fmax3(c3, sv[j + 6], sv[j + 7]);
  }
  return fmaxf(fmax3(c0, c1, c2), c3);
}

// P = 2^(s * c - m) of 64 scores as 32 bf16 pairs (key 2k in the low half of pw[k]);
// returns the fp32 sum of the unrounded values.  m = -inf means every score seen so far
// is masked (-inf): the offset is then 0 and every P is 2^-inf = 0.  Packed fp32x2 FMA
// and add halve their instruction count.
__device__ __forceinline__ float exp_p64(const float (&sv)[64], float c, float m, uint32_t (&pw)[32]) {
  const float nm = m == -INFINITY ? 0.f : -m;
  const float2 cc = make_float2(c, c), nm2 = make_float2(nm, nm);
  float2 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float2 t = __ffma2_rn(make_float2(sv[2 * k], sv[2 * k + 1]), cc, nm2);
    const float e0 = ptx::ex2(t.x), e1 = ptx::ex2(t.y);
    acc[k & 3] = __fadd2_rn(acc[k & 3], make_float2(e0, e1));
    pw[k] = ptx::cvt_bf16x2(e0, e1);
  }
  const float2 s2 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return s2.x + s2.y;
}

// 64-bit visibility mask of keys [j0, j0 + 64) for tree node `node` (half a KV tile).
__device__ __forceinline__ uint64_t key_mask(int j0, int P, int N, int node, const int* s_par) {
  if (j0 + 64 <= P) return ~0ull;
  uint64_t vis = 0;
  if (j0 < P) vis = (1ull << (P - j0)) - 1ull;
  int a = node, guard = 0;
  while (a >= 0 && guard <= N) {
    const int j = P + a - j0;
    if (j >= 0 && j < 64) vis |= 1ull << j;
    const int pa = s_par[a];
    if (pa >= a) break;  // malformed (flagged when loaded)
    a = pa;
    ++guard;
  }
  return vis;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, TcArgs a) {
  ptx::griddep_launch_dependents();
  using C = TcCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ float s_xmax[2][2][kRows];  // [tile parity][half][row] partial row maxima
  __shared__ float s_xl[2][kRows];       // [half][row] partial row sums
  const uint32_t mis = ptx::smem_addr(smem_raw) & 1023u;
  unsigned char* sm = smem_raw + ((1024u - mis) & 1023u);
  unsigned char* sQ = sm + C::kOffQ;
  unsigned char* sK = sm + C::kOffK;
  unsigned char* sV = sm + C::kOffV;
  int* s_par = reinterpret_cast<int*>(sm + C::kOffPar);
  Bars* bars = reinterpret_cast<Bars*>(sm + C::kOffBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the splits of one row tile are consecutive in x and form one cluster (rank = split)
  const int mt = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int i0 = mt * a.NT;
  const int rows_used = a.G * a.NT;
  __shared__ int s_wfirst[kThreads / 32];  // per warp: first padding row it saw (or N)

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kKSlots; ++s) {
      ptx::mbar_init(&bars->k_full[s], 1);
      ptx::mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      ptx::mbar_init(&bars->v_full[s], 1);
      ptx::mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars->s_full[s], 1);
      ptx::mbar_init(&bars->s_free[s], 8);
      ptx::mbar_init(&bars->p_full[s], 8);
      ptx::mbar_init(&bars->pv_done[s], 1);
    }
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->s_done, 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {  // kernel parameters: safe before the wait
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  // the set-up above touches only shared memory, TMEM and parameters, so it overlaps the
  // previous kernel's tail (programmatic dependent launch); global memory after this
  ptx::griddep_wait();
  if (warp >= 2) {
    // parent array for the mask; zero the Q rows that no TMA box fills
    const int t = threadIdx.x - 64;
    int bad = 0, first_pad = a.N;
    for (int c = t; c < a.N; c += kThreads - 64) {
      const int p = a.parent[(size_t)b * a.N + c];
      s_par[c] = p;
      // trailing padding rows of a ragged batch hold parent -1; an active row must not
      // follow one
      const bool prev_pad = c >= 2 && a.parent[(size_t)b * a.N + c - 1] == -1;
      if (!((c == 0) ? (p == -1) : (p == -1 || (p >= 0 && p < c && !prev_pad)))) bad = 1;
      if (c > 0 && p == -1) first_pad = min(first_pad, c);
    }
    first_pad = __reduce_min_sync(0xffffffffu, first_pad);
    if (lane == 0) s_wfirst[warp] = first_pad;
    if (bad) set_dev_status(a.dev_status, TV_DEV_BAD_TREE);
    for (int r = rows_used + t; r < kRows; r += kThreads - 64)
      for (int db = 0; db < C::kDB; ++db) {
        uint4* row = reinterpret_cast<uint4*>(sQ + db * C::kQBlock + r * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
      }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // active rows 0..n_act-1 (a ragged batch pads with parent -1): keys and row tiles past
  // them are never needed
  int n_act = a.N;
#pragma unroll
  for (int w = 2; w < kThreads / 32; ++w) n_act = min(n_act, s_wfirst[w]);
  const int nodes_hi = min(n_act, i0 + a.NT);
  const int t_all = i0 < n_act ? (a.P + nodes_hi + kBN - 1) / kBN : 0;
  const int tps = (t_all + a.splits - 1) / a.splits;
  const int t_begin = split * tps;
  const int nt = max(0, min(t_all, t_begin + tps) - t_begin);

  if (warp == 0) {
    // ------------------------------------------------------------------ producers
    if (lane == 0 && nt > 0) {
      // Q once, then the K tiles; a slot is refilled once S of its previous tile is done
      int issued[kKSlots];
#pragma unroll
      for (int s = 0; s < kKSlots; ++s) issued[s] = 0;
      ptx::mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(rows_used * 128 * C::kDB));
      for (int g = 0; g < a.G; ++g)
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(sQ + db * C::kQBlock + g * a.NT * 128, &tmQ, &bars->q_full, db * 64, i0,
                           b * a.Hq + hk * a.G + g);
      for (int t = 0; t < nt; ++t) {
        const int ks = t % kKSlots;
        if (t >= kKSlots && !ptx::mbar_wait(&bars->k_empty[ks], ((t / kKSlots) - 1) & 1, abort_flag)) break;
        unsigned char* dst = sK + ks * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN;
        ptx::mbar_arrive_expect_tx(&bars->k_full[ks], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(dst + db * C::kKVBlock, &tmK, &bars->k_full[ks], db * 64, j0, b * a.Hkv + hk);
        ++issued[ks];
      }
      // never leave the CTA with copies in flight
      ptx::mbar_wait(&bars->q_full, 0, abort_flag);
      for (int s = 0; s < kKSlots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->k_full[s], (issued[s] - 1) & 1, abort_flag);
    } else if (lane == 1 && nt > 0) {
      // the V tiles; a slot is refilled once PV of its previous tile is done
      int issued[kVSlots];
#pragma unroll
      for (int s = 0; s < kVSlots; ++s) issued[s] = 0;
      for (int t = 0; t < nt; ++t) {
        const int vs = t % kVSlots;
        if (t >= kVSlots && !ptx::mbar_wait(&bars->v_empty[vs], ((t / kVSlots) - 1) & 1, abort_flag)) break;
        unsigned char* dst = sV + vs * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN;
        ptx::mbar_arrive_expect_tx(&bars->v_full[vs], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(dst + db * C::kKVBlock, &tmV, &bars->v_full[vs], db * 64, j0, b * a.Hkv + hk);
        ++issued[vs];
      }
      for (int s = 0; s < kVSlots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->v_full[s], (issued[s] - 1) & 1, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (nt > 0 && ptx::mbar_wait(&bars->q_full, 0, abort_flag)) {
        constexpr uint32_t idS = ptx::idesc_bf16(kRows, kBN, false, false);
        const uint32_t qaddr = ptx::smem_addr(sQ);
        bool ok = true;
        auto issue_s = [&](int t) -> bool {
          const int ks = t % kKSlots, sb = t & 1;
          if (!ptx::mbar_wait(&bars->k_full[ks], (t / kKSlots) & 1, abort_flag)) return false;
          if (t >= 2 && !ptx::mbar_wait(&bars->s_free[sb], ((t >> 1) - 1) & 1, abort_flag)) return false;
          ptx::tc_fence_after();
          const uint32_t kaddr = ptx::smem_addr(sK + ks * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;  // 16-element K step inside a 128-byte row
            const uint64_t ad = ptx::sdesc_sw128(qaddr + (kk >> 2) * C::kQBlock + off, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * C::kKVBlock + off, 16, 1024);
            ptx::mma_bf16_ss(tmem + sb * kBN, ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&bars->s_full[sb]);
          ptx::mma_commit(&bars->k_empty[ks]);
          return true;
        };
        // S = QK^T tiles run ahead of the softmax (bounded by the two S buffers); the PV
        // products are issued by warp 10, so neither waits behind the other's issue
        for (int t = 0; ok && t < nt; ++t) ok = issue_s(t);
      }
      ptx::mma_commit(&bars->s_done);
      ptx::mbar_wait(&bars->s_done, 0, abort_flag);
    }
    __syncwarp();
  } else if (warp == kThreads / 32 - 1) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0) {
      if (nt > 0) {
        constexpr uint32_t idO = ptx::idesc_bf16(kRows, D, false, true);
        for (int t = 0; t < nt; ++t) {
          const int vs = t % kVSlots, pb = t & 1;
          if (!ptx::mbar_wait(&bars->p_full[pb], (t >> 1) & 1, abort_flag)) break;
          if (!ptx::mbar_wait(&bars->v_full[vs], (t / kVSlots) & 1, abort_flag)) break;
          ptx::tc_fence_after();
          const uint32_t vaddr = ptx::smem_addr(sV + vs * C::kTileBytes);
          const uint32_t paddr = tmem + C::kColP + pb * (kBN / 2);  // 16 keys = 8 columns
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t bd = ptx::sdesc_sw128(vaddr + kk * 16 * 128, C::kKVBlock, 1024);
            ptx::mma_bf16_ts(tmem + C::kColO, paddr + kk * 8, bd, idO, (t > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&bars->v_empty[vs]);
          ptx::mma_commit(&bars->pv_done[pb]);
        }
      }
      ptx::mma_commit(&bars->o_done);
      ptx::mbar_wait(&bars->o_done, 0, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax rows
    // two threads per row: warps 2-5 take keys [0, 64) of each tile, warps 6-9 keys
    // [64, 128) (warp w and w + 4 read the same TMEM lane quarter); the halves agree on the
    // row max through shared memory and a barrier of the warp pair once per tile
    const int q4 = warp & 3;
    const int h = (warp - 2) >> 2;
    const int r = q4 * 32 + lane;
    const int g = r / a.NT, il = r % a.NT;
    const int node = i0 + il;
    const bool valid = (g < a.G) && (node < a.N) && (r < rows_used) && !(node > 0 && s_par[node] == -1);
    const int mnode = valid ? node : 0;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int c_lo = h * (kBN / 2);  // this thread's key columns in a tile
    const int d_lo = h * (D / 2);    // and its O columns
    const uint32_t pair_bar = 1 + q4;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // after a failed wait the loop keeps running without waiting or computing, so that
    // both threads of a row still meet at every pair barrier
    for (int t = 0; t < nt; ++t) {
      const int sb = t & 1;
      if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->s_full[sb], (t >> 1) & 1, abort_flag));
      float sv[kBN / 2];
      if (ok) {
        ptx::tc_fence_after();
        ptx::tmem_ld32(tmem + lane_base + sb * kBN + c_lo, sv);
        ptx::tmem_ld32(tmem + lane_base + sb * kBN + c_lo + 32, sv + 32);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->s_free[sb]);
      } else {
#pragma unroll
        for (int j = 0; j < kBN / 2; ++j) sv[j] = -INFINITY;
      }

      const int j0 = (t_begin + t) * kBN;
      const uint64_t vis = key_mask(j0 + c_lo, a.P, a.N, mnode, s_par);
      if (vis != ~0ull) {  // tree / tail tiles: hidden keys become -inf (exp -> 0)
#pragma unroll
        for (int j = 0; j < kBN / 2; ++j)
          if (!((vis >> j) & 1ull)) sv[j] = -INFINITY;
      }
      float tm = max64(sv, -INFINITY);
      s_xmax[t & 1][h][r] = tm;
      pair_sync();
      tm = fmaxf(tm, s_xmax[t & 1][h ^ 1][r]);
      const float tms = tm * a.c;
      float alpha = 1.f;
      bool need = false;
      if (tms > m_run + kRescaleLog2) {
        if (m_run != -INFINITY) {
          alpha = ptx::ex2(m_run - tms);
          need = true;
        }
        m_run = tms;
      }
      if (__any_sync(0xffffffffu, need) && t > 0 && ok) {
        // O already holds PV(t-1): wait for it, then scale this thread's half of the row
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag));
      }
      if (__any_sync(0xffffffffu, need) && t > 0 && ok) {
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          float ov[32];
          ptx::tmem_ld32(tmem + lane_base + C::kColO + d_lo + c0, ov);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] *= alpha;
          ptx::tmem_st32(tmem + lane_base + C::kColO + d_lo + c0, ov);
        }
        ptx::tmem_wait_st();
      }
      l_run *= alpha;
      // P buffer t & 1 is free once PV(t-2) has completed
      if (t >= 2 && ok)
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->pv_done[sb], ((t >> 1) - 1) & 1, abort_flag));
      if (!ok) continue;  // nothing more to compute or signal for this tile
      // P = 2^(S*c - m_run) on visible keys, bf16 pairs along the key axis, into this
      // thread's 32 columns of the TMEM P buffer (its row's lane)
      uint32_t pw[kBN / 4];
      l_run += exp_p64(sv, a.c, m_run, pw);
      ptx::tmem_st32u(tmem + lane_base + C::kColP + sb * (kBN / 2) + h * (kBN / 4), pw);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->p_full[sb]);
    }
    // ---- epilogue: the row's sum is the two halves' sums
    s_xl[h][r] = l_run;
    pair_sync();
    l_run += s_xl[h ^ 1][r];
    bool have_o = false;
    if (nt > 0) {
      ok = ptx::mbar_wait(&bars->o_done, 0, abort_flag) && ok;
      ok = __all_sync(0xffffffffu, ok);
      have_o = ok;
      if (ok) ptx::tc_fence_after();
    }
    const int hh = hk * a.G + g;
    const size_t orow = (((size_t)b * a.Hq + hh) * a.N + node) * D;
    if (a.splits == 1) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(tmem + lane_base + C::kColO + d_lo + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + d_lo + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = ptx::cvt_bf16x2(ov[8 * k + 0] * inv, ov[8 * k + 1] * inv);
            u.y = ptx::cvt_bf16x2(ov[8 * k + 2] * inv, ov[8 * k + 3] * inv);
            u.z = ptx::cvt_bf16x2(ov[8 * k + 4] * inv, ov[8 * k + 5] * inv);
            u.w = ptx::cvt_bf16x2(ov[8 * k + 6] * inv, ov[8 * k + 7] * inv);
            dst[k] = u;
          }
        }
      }
    } else {
      // park this split's unnormalised O as row-major [128][D] fp32 with the 16-byte chunks
      // of row r XOR-swizzled by (r & 7) (conflict-free 16-byte stores), plus (m, l), in
      // the drained K/V ring for the cluster merge below
      unsigned char* part = sK;
      float2* ml = reinterpret_cast<float2*>(sK + D * kRows * 4);
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(tmem + lane_base + C::kColO + d_lo + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int chunk = (d_lo + c0) / 4 + k;
          *reinterpret_cast<float4*>(part + r * D * 4 + ((chunk ^ (r & 7)) << 4)) =
              make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
        }
      }
      if (h == 0) ml[r] = make_float2(have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
    }
    ptx::tc_fence_before();
  }
  __syncwarp();
  if (a.splits > 1) {
    // The KV splits of this row tile form one thread-block cluster.  After every CTA has
    // parked its partial, CTA `split` merges rows [split*R, split*R + R) by reading all
    // peers' partials through distributed shared memory, then nobody leaves before every
    // peer has finished reading.
    ptx::cluster_sync();
    {
      // every thread; item = (row of this CTA's slice, 16-byte chunk of 4 columns):
      // a warp reads one contiguous row of each peer's partial, all loads issued first
      const int S = a.splits;
      const int R = (kRows + S - 1) / S;
      const int r0 = split * R, r1 = min(kRows, r0 + R);
      const int nrows = max(0, r1 - r0);
      constexpr int kChunks = D / 4;
      const uint32_t part_local = ptx::smem_addr(sK);
      const uint32_t ml_local = ptx::smem_addr(sK + D * kRows * 4);
      for (int item = threadIdx.x; item < nrows * kChunks; item += kThreads) {
        const int rr = r0 + item / kChunks;
        const int ch = item % kChunks;
        const int gg = rr / a.NT, ii = i0 + rr % a.NT;
        if (gg >= a.G || ii >= a.N || rr >= rows_used || (ii > 0 && s_par[ii] == -1)) continue;
        float2 mlv[kMaxSplits];
        float4 x[kMaxSplits];
        const uint32_t moff = (uint32_t)(rr * 8);
        const uint32_t xoff = (uint32_t)(rr * D * 4 + ((ch ^ (rr & 7)) << 4));
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S) {
            mlv[s2] = ptx::ld_cluster_f32x2(ptx::map_cluster(ml_local, s2) + moff);
            x[s2] = ptx::ld_cluster_f32x4(ptx::map_cluster(part_local, s2) + xoff);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2)
          if (s2 < S) M = fmaxf(M, mlv[s2].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S && mlv[s2].x != -INFINITY) {
            const float w = ptx::ex2(mlv[s2].x - M);
            L = fmaf(mlv[s2].y, w, L);
            acc.x = fmaf(w, x[s2].x, acc.x);
            acc.y = fmaf(w, x[s2].y, acc.y);
            acc.z = fmaf(w, x[s2].z, acc.z);
            acc.w = fmaf(w, x[s2].w, acc.w);
          }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t o2 = (((size_t)b * a.Hq + hk * a.G + gg) * a.N + ii) * D + ch * 4;
        uint2 u;
        u.x = ptx::cvt_bf16x2(acc.x * inv, acc.y * inv);
        u.y = ptx::cvt_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + o2) = u;
      }
    }
    __syncwarp();
    ptx::cluster_sync();
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// Paired row tiles.  One CTA owns two 128-row tiles A and B of the same (b, kv head)
// (tiles 2m and 2m + 1) and streams the KV range once for both: every K/V tile fetched
// serves 256 query rows.  The two tiles ping-pong on the tensor core: while the softmax
// warps of tile A turn S_A into probabilities, the tensor core runs S_B and PV_B, and
// the other way round.
//   warp 0      TMA producers: lane 0 loads Q_A, Q_B once, then K tiles into a 2-slot
//               ring; lane 1 loads the V tiles into a 2-slot ring
//   warp 1      TMEM owner; lane 0 issues S_X = Q_X K_t^T for X = A, B
//   warps 2..5  softmax of tile A, warps 6..9 softmax of tile B: one thread per row
//               (TMEM lane), 128 keys per tile, no partner thread to wait for
//   warp 10     lane 0 issues O_X += P_X V_t
// TMEM columns: S_A 0..127, S_B 128..255, O_A 256.., O_B 384...  P_X (bf16) is written
// over S_X by its own row's thread: keys 64..127 into columns 64..95 (S values already
// in registers), then keys 0..63 into columns 0..31 after they have been read again.
// S_X of the next KV tile is issued only once PV_X of the current one has completed, so
// it never overwrites P_X early, and O_X is quiescent whenever its softmax runs.
constexpr int kPairSlots = 2;  // K ring and V ring depth

template <int D>
struct PairCfg {
  static constexpr int kDB = D / 64;
  static constexpr int kQBlock = kRows * 128;       // bytes per column block of one Q tile
  static constexpr int kQTile = kDB * kQBlock;      // one Q tile
  static constexpr int kKVBlock = kBN * 128;        // bytes per column block of a K or V tile
  static constexpr int kTileBytes = kDB * kKVBlock; // one K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + kPairSlots * kTileBytes;
  static constexpr int kOffPar = kOffV + kPairSlots * kTileBytes;
  static constexpr int kOffBar = kOffPar + kMaxNodes * 4;
  static constexpr int kSmemUsed = kOffBar + 256;
  static constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 2 * kBN;           // O_X at kColO + X * 128
  static_assert(kColO + kBN + D <= kTmemCols, "TMEM budget");
  static_assert(2 * kPairSlots * kTileBytes >= 2 * kRows * D * 4, "split partials fit in the drained rings");
  static_assert(2 * kQTile >= 2 * kRows * 8, "(m, l) of both tiles fit in the drained Q tiles");
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
};

struct PairBars {
  uint64_t q_full;
  uint64_t k_full[kPairSlots];
  uint64_t k_empty[kPairSlots];
  uint64_t v_full[kPairSlots];
  uint64_t v_empty[kPairSlots];
  uint64_t s_full[2];   // S_X(t) complete
  uint64_t p_full[2];   // P_X(t) written (4 warps)
  uint64_t pv_done[2];  // PV_X(t) complete
  uint64_t o_done;
  uint64_t s_done;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, TcArgs a) {
  ptx::griddep_launch_dependents();
  using C = PairCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t mis = ptx::smem_addr(smem_raw) & 1023u;
  unsigned char* sm = smem_raw + ((1024u - mis) & 1023u);
  unsigned char* sQ = sm + C::kOffQ;
  unsigned char* sK = sm + C::kOffK;
  unsigned char* sV = sm + C::kOffV;
  int* s_par = reinterpret_cast<int*>(sm + C::kOffPar);
  PairBars* bars = reinterpret_cast<PairBars*>(sm + C::kOffBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the splits of one tile pair are consecutive in x and form one cluster (rank = split)
  const int mp = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  const int hk = blockIdx.y, b = blockIdx.z;
  int i0[2], t_allx[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    i0[x] = (2 * mp + x) * a.NT;
    t_allx[x] = i0[x] < a.N ? (a.P + min(a.N, i0[x] + a.NT) + kBN - 1) / kBN : 0;
  }
  const int t_all = max(t_allx[0], t_allx[1]);
  const int tps = (t_all + a.splits - 1) / a.splits;
  const int t_begin = split * tps;
  int ntx[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) ntx[x] = max(0, min(t_allx[x], t_begin + tps) - t_begin);
  const int nt = max(ntx[0], ntx[1]);
  const int rows_used = a.G * a.NT;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kPairSlots; ++s) {
      ptx::mbar_init(&bars->k_full[s], 1);
      ptx::mbar_init(&bars->k_empty[s], 1);
      ptx::mbar_init(&bars->v_full[s], 1);
      ptx::mbar_init(&bars->v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(&bars->s_full[x], 1);
      ptx::mbar_init(&bars->p_full[x], 4);
      ptx::mbar_init(&bars->pv_done[x], 1);
    }
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->s_done, 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {  // kernel parameters: safe before the wait
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  // the set-up above touches only shared memory, TMEM and parameters, so it overlaps the
  // previous kernel's tail (programmatic dependent launch); global memory after this
  ptx::griddep_wait();
  if (warp >= 2) {
    // parent array for the mask; zero the Q rows that no TMA box fills
    const int t = threadIdx.x - 64;
    int bad = 0;
    for (int c = t; c < a.N; c += kThreads - 64) {
      const int p = a.parent[(size_t)b * a.N + c];
      s_par[c] = p;
      // trailing padding rows of a ragged batch hold parent -1; an active row must not
      // follow one
      const bool prev_pad = c >= 2 && a.parent[(size_t)b * a.N + c - 1] == -1;
      if (!((c == 0) ? (p == -1) : (p == -1 || (p >= 0 && p < c && !prev_pad)))) bad = 1;
    }
    if (bad) set_dev_status(a.dev_status, TV_DEV_BAD_TREE);
    for (int r = rows_used + t; r < 2 * kRows; r += kThreads - 64) {
      const int x = r >= kRows ? 1 : 0, rr = r - x * kRows;
      if (rr < rows_used) continue;
      for (int db = 0; db < C::kDB; ++db) {
        uint4* row = reinterpret_cast<uint4*>(sQ + x * C::kQTile + db * C::kQBlock + rr * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
      }
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ producers
    if (lane == 0 && nt > 0) {
      int issued[kPairSlots] = {0, 0};
      uint32_t qbytes = 0;
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (ntx[x] > 0) qbytes += (uint32_t)(rows_used * 128 * C::kDB);
      ptx::mbar_arrive_expect_tx(&bars->q_full, qbytes);
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (ntx[x] > 0)
          for (int g = 0; g < a.G; ++g)
            for (int db = 0; db < C::kDB; ++db)
              ptx::tma_load_3d(sQ + x * C::kQTile + db * C::kQBlock + g * a.NT * 128, &tmQ, &bars->q_full, db * 64,
                               i0[x], b * a.Hq + hk * a.G + g);
      for (int t = 0; t < nt; ++t) {
        const int ks = t % kPairSlots;
        if (t >= kPairSlots && !ptx::mbar_wait(&bars->k_empty[ks], ((t / kPairSlots) - 1) & 1, abort_flag)) break;
        unsigned char* dst = sK + ks * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN;
        ptx::mbar_arrive_expect_tx(&bars->k_full[ks], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(dst + db * C::kKVBlock, &tmK, &bars->k_full[ks], db * 64, j0, b * a.Hkv + hk);
        ++issued[ks];
      }
      // never leave the CTA with copies in flight
      ptx::mbar_wait(&bars->q_full, 0, abort_flag);
      for (int s = 0; s < kPairSlots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->k_full[s], (issued[s] - 1) & 1, abort_flag);
    } else if (lane == 1 && nt > 0) {
      int issued[kPairSlots] = {0, 0};
      for (int t = 0; t < nt; ++t) {
        const int vs = t % kPairSlots;
        if (t >= kPairSlots && !ptx::mbar_wait(&bars->v_empty[vs], ((t / kPairSlots) - 1) & 1, abort_flag)) break;
        unsigned char* dst = sV + vs * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN;
        ptx::mbar_arrive_expect_tx(&bars->v_full[vs], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db)
          ptx::tma_load_3d(dst + db * C::kKVBlock, &tmV, &bars->v_full[vs], db * 64, j0, b * a.Hkv + hk);
        ++issued[vs];
      }
      for (int s = 0; s < kPairSlots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->v_full[s], (issued[s] - 1) & 1, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S issuer
    if (lane == 0) {
      if (nt > 0 && ptx::mbar_wait(&bars->q_full, 0, abort_flag)) {
        constexpr uint32_t idS = ptx::idesc_bf16(kRows, kBN, false, false);
        bool ok = true;
        for (int t = 0; ok && t < nt; ++t) {
          const int ks = t % kPairSlots;
          if (!ptx::mbar_wait(&bars->k_full[ks], (t / kPairSlots) & 1, abort_flag)) break;
          const uint32_t kaddr = ptx::smem_addr(sK + ks * C::kTileBytes);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (t >= ntx[x]) continue;
            // S_X(t) overwrites P_X(t - 1): wait for PV_X(t - 1)
            if (t >= 1 && !ptx::mbar_wait(&bars->pv_done[x], (t - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t qaddr = ptx::smem_addr(sQ + x * C::kQTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;  // 16-element K step inside a 128-byte row
              const uint64_t ad = ptx::sdesc_sw128(qaddr + (kk >> 2) * C::kQBlock + off, 16, 1024);
              const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * C::kKVBlock + off, 16, 1024);
              ptx::mma_bf16_ss(tmem + x * kBN, ad, bd, idS, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(&bars->s_full[x]);
          }
          if (ok) ptx::mma_commit(&bars->k_empty[ks]);
        }
      }
      ptx::mma_commit(&bars->s_done);
      ptx::mbar_wait(&bars->s_done, 0, abort_flag);
    }
    __syncwarp();
  } else if (warp == kThreads / 32 - 1) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t idO = ptx::idesc_bf16(kRows, D, false, true);
      bool ok = true;
      for (int t = 0; ok && t < nt; ++t) {
        const int vs = t % kPairSlots;
        if (!ptx::mbar_wait(&bars->v_full[vs], (t / kPairSlots) & 1, abort_flag)) break;
        const uint32_t vaddr = ptx::smem_addr(sV + vs * C::kTileBytes);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (t >= ntx[x]) continue;
          if (!ptx::mbar_wait(&bars->p_full[x], t & 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t pcol = tmem + x * kBN;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            // keys 0..63 in columns 0..31, keys 64..127 in columns 64..95 (8 columns per 16 keys)
            const uint32_t pa = pcol + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            const uint64_t bd = ptx::sdesc_sw128(vaddr + kk * 16 * 128, C::kKVBlock, 1024);
            ptx::mma_bf16_ts(tmem + C::kColO + x * kBN, pa, bd, idO, (t > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&bars->pv_done[x]);
        }
        if (ok) ptx::mma_commit(&bars->v_empty[vs]);
      }
      ptx::mma_commit(&bars->o_done);
      ptx::mbar_wait(&bars->o_done, 0, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax rows
    const int x = (warp - 2) >> 2;  // tile
    const int q4 = warp & 3;        // TMEM lane quarter of this warp
    const int r = q4 * 32 + lane;
    const int g = r / a.NT, il = r % a.NT;
    const int node = i0[x] + il;
    const bool valid = (g < a.G) && (node < a.N) && (r < rows_used) && !(node > 0 && s_par[node] == -1);
    const int mnode = valid ? node : 0;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t colS = tmem + lane_base + x * kBN;
    const uint32_t colO = tmem + lane_base + C::kColO + x * kBN;
    const int ntm = ntx[x];
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntm; ++t) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->s_full[x], t & 1, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      const int j0 = (t_begin + t) * kBN;
      const uint64_t vis_lo = key_mask(j0, a.P, a.N, mnode, s_par);
      const uint64_t vis_hi = key_mask(j0 + 64, a.P, a.N, mnode, s_par);
      float sv[64];
      // row max over the tile: keys 0..63, then keys 64..127 (kept in registers)
      ptx::tmem_ld32(colS, sv);
      ptx::tmem_ld32(colS + 32, sv + 32);
      ptx::tmem_wait_ld();
      if (vis_lo != ~0ull) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((vis_lo >> j) & 1ull)) sv[j] = -INFINITY;
      }
      float tm = max64(sv, -INFINITY);
      ptx::tmem_ld32(colS + 64, sv);
      ptx::tmem_ld32(colS + 96, sv + 32);
      ptx::tmem_wait_ld();
      if (vis_hi != ~0ull) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((vis_hi >> j) & 1ull)) sv[j] = -INFINITY;
      }
      tm = max64(sv, tm);
      const float tms = tm * a.c;
      float alpha = 1.f;
      bool need = false;
      if (tms > m_run + kRescaleLog2) {
        if (m_run != -INFINITY) {
          alpha = ptx::ex2(m_run - tms);
          need = true;
        }
        m_run = tms;
      }
      if (__any_sync(0xffffffffu, need)) {
        // O_X holds PV_X(t - 1), complete (S_X(t) was issued after it); the wait returns
        // at once and orders the TMEM reads after the MMA's writes
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->pv_done[x], (t - 1) & 1, abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float ov[32];
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] *= alpha;
          ptx::tmem_st32(colO + c0, ov);
        }
        ptx::tmem_wait_st();
      }
      l_run *= alpha;
      uint32_t pw[32];
      // P for keys 64..127 over their own S columns 64..95
      float lsum = exp_p64(sv, a.c, m_run, pw);
      ptx::tmem_st32u(colS + 64, pw);
      // keys 0..63 again, then P over columns 0..31
      ptx::tmem_ld32(colS, sv);
      ptx::tmem_ld32(colS + 32, sv + 32);
      ptx::tmem_wait_ld();
      if (vis_lo != ~0ull) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((vis_lo >> j) & 1ull)) sv[j] = -INFINITY;
      }
      lsum += exp_p64(sv, a.c, m_run, pw);
      ptx::tmem_st32u(colS, pw);
      l_run += lsum;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->p_full[x]);
    }
    // ---- epilogue: every MMA of the CTA (both tiles) is complete at o_done, so the
    // rings may be reused for the split partials
    bool have_o = false;
    if (nt > 0) {
      const bool done = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->o_done, 0, abort_flag));
      have_o = done && ok && ntm > 0;
      if (done) ptx::tc_fence_after();
    }
    const int hh = hk * a.G + g;
    const size_t orow = (((size_t)b * a.Hq + hh) * a.N + node) * D;
    if (a.splits == 1) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = ptx::cvt_bf16x2(ov[8 * k + 0] * inv, ov[8 * k + 1] * inv);
            u.y = ptx::cvt_bf16x2(ov[8 * k + 2] * inv, ov[8 * k + 3] * inv);
            u.z = ptx::cvt_bf16x2(ov[8 * k + 4] * inv, ov[8 * k + 5] * inv);
            u.w = ptx::cvt_bf16x2(ov[8 * k + 6] * inv, ov[8 * k + 7] * inv);
            dst[k] = u;
          }
        }
      }
    } else {
      // park the unnormalised O of row R = x * 128 + r as row-major [256][D] fp32 with
      // the 16-byte chunks XOR-swizzled by (R & 7), over the drained K and V rings, and
      // (m, l) over the drained Q tiles
      const int R = x * kRows + r;
      unsigned char* part = sK;
      float2* ml = reinterpret_cast<float2*>(sQ);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int chunk = c0 / 4 + k;
          *reinterpret_cast<float4*>(part + (size_t)R * D * 4 + ((chunk ^ (R & 7)) << 4)) =
              make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
        }
      }
      ml[R] = make_float2(have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
    }
    ptx::tc_fence_before();
  }
  __syncwarp();
  if (a.splits > 1) {
    // merge as in attn_tc_kernel, over the 256 rows of the pair
    ptx::cluster_sync();
    {
      const int S = a.splits;
      constexpr int kPRows = 2 * kRows;
      const int R = (kPRows + S - 1) / S;
      const int r0 = split * R, r1 = min(kPRows, r0 + R);
      const int nrows = max(0, r1 - r0);
      constexpr int kChunks = D / 4;
      const uint32_t part_local = ptx::smem_addr(sK);
      const uint32_t ml_local = ptx::smem_addr(sQ);
      for (int item = threadIdx.x; item < nrows * kChunks; item += kThreads) {
        const int rr = r0 + item / kChunks;
        const int ch = item % kChunks;
        const int xx = rr >= kRows ? 1 : 0, rt = rr - xx * kRows;
        const int gg = rt / a.NT, ii = i0[xx] + rt % a.NT;
        if (gg >= a.G || ii >= a.N || rt >= rows_used || (ii > 0 && s_par[ii] == -1)) continue;
        float2 mlv[kMaxSplits];
        float4 xv[kMaxSplits];
        const uint32_t moff = (uint32_t)(rr * 8);
        const uint32_t xoff = (uint32_t)(rr * D * 4 + ((ch ^ (rr & 7)) << 4));
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S) {
            mlv[s2] = ptx::ld_cluster_f32x2(ptx::map_cluster(ml_local, s2) + moff);
            xv[s2] = ptx::ld_cluster_f32x4(ptx::map_cluster(part_local, s2) + xoff);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2)
          if (s2 < S) M = fmaxf(M, mlv[s2].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S && mlv[s2].x != -INFINITY) {
            const float w = ptx::ex2(mlv[s2].x - M);
            L = fmaf(mlv[s2].y, w, L);
            acc.x = fmaf(w, xv[s2].x, acc.x);
            acc.y = fmaf(w, xv[s2].y, acc.y);
            acc.z = fmaf(w, xv[s2].z, acc.z);
            acc.w = fmaf(w, xv[s2].w, acc.w);
          }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t o2 = (((size_t)b * a.Hq + hk * a.G + gg) * a.N + ii) * D + ch * 4;
        uint2 u;
        u.x = ptx::cvt_bf16x2(acc.x * inv, acc.y * inv);
        u.y = ptx::cvt_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + o2) = u;
      }
    }
    __syncwarp();
    ptx::cluster_sync();
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// Paired row tiles with 64-key KV tiles and two S buffers per row tile.  The same roles
// as attn_pair_kernel, but with 64-key tiles each tile's S takes 64 TMEM columns, so both
// row tiles get two S buffers next to their O accumulators: S_X of KV tile t + 1 is
// computed while the softmax of tile t runs, and the tensor core no longer waits for the
// serial S -> softmax -> PV chain of each tile.  P_X(t) (bf16, 32 columns) is written over
// the first half of its own S buffer by its row's thread; S_X(t + 2) reuses that buffer
// once PV_X(t) has completed.  Each row tile has its own S issuing thread: one thread
// issues an N = 64 product with both operands in shared memory only every ~100 cycles
// (37 cycles of tensor work), so a single issuer for both tiles left the tensor core
// waiting; two issuers took the long-context attention from 475 to 407 us.
// TMEM columns: S_A[0] 0..63, S_A[1] 64..127, S_B[0] 128..191, S_B[1] 192..255,
// O_A 256.., O_B 384...
// Warps: 0 TMA producers (lane 0 Q and K, lane 1 V), 1 S issuer of tile A and TMEM owner,
// 2-9 softmax (four per tile, one thread per row), 10 PV issuer, 11 S issuer of tile B.
constexpr int kBN2 = 64;       // keys per KV tile
constexpr int kPair2Slots = 4; // K ring and V ring depth
constexpr int kP2Threads = 384;  // 12 warps

template <int D>
struct Pair2Cfg {
  static constexpr int kDB = D / 64;
  static constexpr int kQBlock = kRows * 128;        // bytes per column block of one Q tile
  static constexpr int kQTile = kDB * kQBlock;
  static constexpr int kKVBlock = kBN2 * 128;        // bytes per column block of a K or V tile
  static constexpr int kTileBytes = kDB * kKVBlock;  // one K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + kPair2Slots * kTileBytes;
  static constexpr int kOffPar = kOffV + kPair2Slots * kTileBytes;
  static constexpr int kOffBar = kOffPar + kMaxNodes * 4;
  static constexpr int kSmemUsed = kOffBar + 512;
  static constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;               // O_X at kColO + X * 128
  static_assert(kColO + kRows + D <= kTmemCols, "TMEM budget");
  static_assert(2 * kPair2Slots * kTileBytes >= 2 * kRows * D * 4, "split partials fit in the drained rings");
  static_assert(2 * kQTile >= 2 * kRows * 8, "(m, l) of both tiles fit in the drained Q tiles");
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
};

struct Pair2Bars {
  uint64_t q_full;
  uint64_t k_full[kPair2Slots];
  uint64_t k_empty[kPair2Slots];
  uint64_t v_full[kPair2Slots];
  uint64_t v_empty[kPair2Slots];
  uint64_t s_full[2][2];   // [row tile][S buffer]: S_X(t) complete, t & 1 == buffer
  uint64_t p_full[2][2];   // P_X(t) written (4 warps)
  uint64_t pv_done[2][2];  // PV_X(t) complete
  uint64_t o_done;
  uint64_t s_done[2];
  uint32_t tmem_base;
  int abort;
};

// One S product of attn_pair2_kernel (D = 128): the 8 MMAs of K = 16 each from one asm
// block, the first overwriting S.  A descriptors come precomputed (the Q tile's never
// change); the K tile's follow from its first one by constant steps in 16-byte units:
// 32 bytes per K step inside a 128-byte row, 8 KB to the second column block.  Issuing
// threads share their SM sub-partitions with softmax warps, so fewer instructions per MMA
// issue the short (N = 64) products sooner.
__device__ __forceinline__ void s_product_d128(uint32_t d, const uint64_t (&ad)[8], uint64_t bd0, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b32 z;\n\tmov.b32 z, 0;\n\tsetp.ne.b32 p0, z, 0;\n\tsetp.eq.b32 p1, z, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, p0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, p1;\n\t}" ::"r"(d),
      "l"(ad[0]), "l"(ad[1]), "l"(ad[2]), "l"(ad[3]), "l"(ad[4]), "l"(ad[5]), "l"(ad[6]), "l"(ad[7]),
      "l"(bd0), "l"(bd0 + 2), "l"(bd0 + 4), "l"(bd0 + 6), "l"(bd0 + 512), "l"(bd0 + 514), "l"(bd0 + 516),
      "l"(bd0 + 518), "r"(idesc)
      : "memory");
}
// One PV product (D = 128, 64 keys): 4 MMAs of K = 16 with P read from TMEM (8 columns per
// 16 keys) and V tile rows 16 apart (2 KB = 128 descriptor units); the first accumulates
// only when acc0 != 0.
__device__ __forceinline__ void pv_product_d128(uint32_t d, uint32_t a, uint64_t vd0, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b32 z;\n\tmov.b32 z, 0;\n\tsetp.ne.b32 p0, %10, 0;\n\tsetp.eq.b32 p1, z, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %9, p0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %9, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %9, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %9, p1;\n\t}" ::"r"(d),
      "r"(a), "r"(a + 8), "r"(a + 16), "r"(a + 24), "l"(vd0), "l"(vd0 + 128), "l"(vd0 + 256), "l"(vd0 + 384),
      "r"(idesc), "r"(acc0)
      : "memory");
}

template <int D, bool kPair>
__global__ void __launch_bounds__(kP2Threads, 1)
    attn_pair2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, TcArgs a) {
  static_assert(!kPair || D == 128, "the SM-pair form splits V into two 64-column blocks");
  ptx::griddep_launch_dependents();
  using C = Pair2Cfg<D>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t mis = ptx::smem_addr(smem_raw) & 1023u;
  unsigned char* sm = smem_raw + ((1024u - mis) & 1023u);
  unsigned char* sQ = sm + C::kOffQ;
  unsigned char* sK = sm + C::kOffK;
  unsigned char* sV = sm + C::kOffV;
  int* s_par = reinterpret_cast<int*>(sm + C::kOffPar);
  Pair2Bars* bars = reinterpret_cast<Pair2Bars*>(sm + C::kOffBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mp = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  const int hk = blockIdx.y, b = blockIdx.z;
  // K/V multicast: the two tile pairs of a cluster each load half of every K and V tile
  // (32 of its 64 rows) into both CTAs' rings; a slot is refilled once both CTAs' products
  // are done with it (their commits arrive on both CTAs' empty barriers)
  const bool mc = !kPair && a.mcast != 0;
  // SM pair (kPair): the two CTAs of a cluster (tile pairs 2c and 2c + 1, one KV head)
  // compute every product as one M = 256 MMA issued by the even CTA: the 128 rows of
  // each CTA's row tile X form half of product X.  Each CTA loads its half of every K tile
  // (32 of the 64 keys, both column blocks) and of every V tile (64 of the 128 value
  // columns); the copies complete on the even CTA's barriers, the MMAs' commits arrive on
  // both CTAs' barriers, and both CTAs' softmax warps report P on the even CTA's barrier.
  const uint32_t crank = (mc || kPair) ? (blockIdx.x & 1u) : 0u;
  const bool issuer_cta = !kPair || crank == 0;
  int i0[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) i0[x] = (2 * mp + x) * a.NT;
  const int rows_used = a.G * a.NT;
  __shared__ int s_wfirst[kP2Threads / 32];  // per warp: first padding row it saw (or N)

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kPair2Slots; ++s) {
      ptx::mbar_init(&bars->k_full[s], 1);
      ptx::mbar_init(&bars->k_empty[s], mc ? 4 : 2);  // both S issuers (of both CTAs)
      ptx::mbar_init(&bars->v_full[s], 1);
      ptx::mbar_init(&bars->v_empty[s], mc ? 2 : 1);
    }
    for (int x = 0; x < 2; ++x)
      for (int u = 0; u < 2; ++u) {
        ptx::mbar_init(&bars->s_full[x][u], 1);
        ptx::mbar_init(&bars->p_full[x][u], kPair ? 8 : 4);  // the softmax warps of tile X (of both CTAs)
        ptx::mbar_init(&bars->pv_done[x][u], 1);
      }
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->s_done[0], 1);
    ptx::mbar_init(&bars->s_done[1], 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(&bars->tmem_base, C::kTmemCols);  // with the peer CTA's warp 1
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&bars->tmem_base, C::kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {  // kernel parameters: safe before the wait
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  // the set-up above touches only shared memory, TMEM and parameters, so it overlaps the
  // previous kernel's tail (programmatic dependent launch); global memory after this
  ptx::griddep_wait();
  if (warp >= 2) {
    const int t = threadIdx.x - 64;
    int bad = 0, first_pad = a.N;
    for (int c = t; c < a.N; c += kP2Threads - 64) {
      const int p = a.parent[(size_t)b * a.N + c];
      s_par[c] = p;
      // trailing padding rows of a ragged batch hold parent -1; an active row must not
      // follow one
      const bool prev_pad = c >= 2 && a.parent[(size_t)b * a.N + c - 1] == -1;
      if (!((c == 0) ? (p == -1) : (p == -1 || (p >= 0 && p < c && !prev_pad)))) bad = 1;
      if (c > 0 && p == -1) first_pad = min(first_pad, c);
    }
    first_pad = __reduce_min_sync(0xffffffffu, first_pad);
    if (lane == 0) s_wfirst[warp] = first_pad;
    if (bad) set_dev_status(a.dev_status, TV_DEV_BAD_TREE);
    for (int r = rows_used + t; r < 2 * kRows; r += kP2Threads - 64) {
      const int x = r >= kRows ? 1 : 0, rr = r - x * kRows;
      if (rr < rows_used) continue;
      for (int db = 0; db < C::kDB; ++db) {
        uint4* row = reinterpret_cast<uint4*>(sQ + x * C::kQTile + db * C::kQBlock + rr * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
      }
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  if (mc || kPair)
    ptx::cluster_sync();  // the peer's barriers are initialised before anything arrives on them
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // active rows 0..n_act-1 (a ragged batch pads with parent -1): keys and row tiles past
  // them are never needed
  int n_act = a.N;
#pragma unroll
  for (int w = 2; w < kP2Threads / 32; ++w) n_act = min(n_act, s_wfirst[w]);
  int t_allx[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    t_allx[x] = i0[x] < n_act ? (a.P + min(n_act, i0[x] + a.NT) + kBN2 - 1) / kBN2 : 0;
    if constexpr (kPair) {  // product X covers row tile X of both CTAs (no KV splits)
      const int i0p = (2 * (mp ^ 1) + x) * a.NT;
      if (i0p < n_act) t_allx[x] = max(t_allx[x], (a.P + min(n_act, i0p + a.NT) + kBN2 - 1) / kBN2);
    }
  }
  const int t_all = max(t_allx[0], t_allx[1]);
  const int tps = (t_all + a.splits - 1) / a.splits;
  const int t_begin = split * tps;
  int ntx[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) ntx[x] = max(0, min(t_allx[x], t_begin + tps) - t_begin);
  const int nt = max(ntx[0], ntx[1]);
  // K/V tiles streamed: with multicast both CTAs of the cluster stream the longer of their
  // two ranges (the other one's extra tiles are loaded and released, never computed)
  int nts = nt;
  if (mc) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int i0p = (2 * (mp ^ 1) + x) * a.NT;
      if (i0p < n_act) nts = max(nts, (a.P + min(n_act, i0p + a.NT) + kBN2 - 1) / kBN2);
    }
  }
  constexpr uint16_t kPairMask = 0x3;

  if (warp == 0) {
    // ------------------------------------------------------------------ producers
    if (lane == 0 && nts > 0) {
      int issued[kPair2Slots] = {0, 0, 0, 0};
      uint32_t qbytes = 0;
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (ntx[x] > 0) qbytes += (uint32_t)(rows_used * 128 * C::kDB);
      // SM pair: both CTAs' Q tiles complete on the even CTA's barrier
      const uint32_t qf = kPair ? ptx::map_cluster(ptx::smem_addr(&bars->q_full), 0) : 0u;
      if (crank == 0 || !kPair) ptx::mbar_arrive_expect_tx(&bars->q_full, kPair ? 2 * qbytes : qbytes);
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (ntx[x] > 0)
          for (int g = 0; g < a.G; ++g)
            for (int db = 0; db < C::kDB; ++db) {
              unsigned char* dq = sQ + x * C::kQTile + db * C::kQBlock + g * a.NT * 128;
              if constexpr (kPair)
                ptx::tma_load_3d_pair(dq, &tmQ, qf, db * 64, i0[x], b * a.Hq + hk * a.G + g);
              else
                ptx::tma_load_3d(dq, &tmQ, &bars->q_full, db * 64, i0[x], b * a.Hq + hk * a.G + g);
            }
      for (int t = 0; t < nts; ++t) {
        const int ks = t % kPair2Slots;
        if (t >= kPair2Slots && !ptx::mbar_wait(&bars->k_empty[ks], ((t / kPair2Slots) - 1) & 1, abort_flag))
          break;
        unsigned char* dst = sK + ks * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN2;
        if constexpr (kPair) {
          // this CTA's 32 keys of the tile, both column blocks (4 KB each); the even CTA
          // expects both halves
          if (crank == 0) ptx::mbar_arrive_expect_tx(&bars->k_full[ks], (uint32_t)C::kTileBytes);
          const uint32_t kf = ptx::map_cluster(ptx::smem_addr(&bars->k_full[ks]), 0);
          for (int db = 0; db < C::kDB; ++db)
            ptx::tma_load_3d_pair(dst + db * (C::kKVBlock / 2), &tmK, kf, db * 64, j0 + (int)crank * (kBN2 / 2),
                                  b * a.Hkv + hk);
          ++issued[ks];
          continue;
        }
        ptx::mbar_arrive_expect_tx(&bars->k_full[ks], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db) {
          if (mc)
            ptx::tma_load_3d_mc(dst + db * C::kKVBlock + crank * (kBN2 / 2) * 128, &tmK, &bars->k_full[ks], db * 64,
                                j0 + (int)crank * (kBN2 / 2), b * a.Hkv + hk, kPairMask);
          else
            ptx::tma_load_3d(dst + db * C::kKVBlock, &tmK, &bars->k_full[ks], db * 64, j0, b * a.Hkv + hk);
        }
        ++issued[ks];
      }
      if constexpr (kPair) {
        // the copies completed on the even CTA's barriers: wait until the products have
        // released the last ones (so that none is in flight at exit); the Q tiles were
        // read by those products
        for (int s = 0; s < kPair2Slots; ++s)
          if (issued[s]) ptx::mbar_wait(&bars->k_empty[s], (issued[s] - 1) & 1, abort_flag);
      } else {
        ptx::mbar_wait(&bars->q_full, 0, abort_flag);
        for (int s = 0; s < kPair2Slots; ++s)
          if (issued[s]) ptx::mbar_wait(&bars->k_full[s], (issued[s] - 1) & 1, abort_flag);
      }
    } else if (lane == 1 && nts > 0) {
      int issued[kPair2Slots] = {0, 0, 0, 0};
      for (int t = 0; t < nts; ++t) {
        const int vs = t % kPair2Slots;
        if (t >= kPair2Slots && !ptx::mbar_wait(&bars->v_empty[vs], ((t / kPair2Slots) - 1) & 1, abort_flag))
          break;
        unsigned char* dst = sV + vs * C::kTileBytes;
        const int j0 = (t_begin + t) * kBN2;
        if constexpr (kPair) {
          // all 64 keys of the tile, this CTA's 64 value columns (one column block)
          if (crank == 0) ptx::mbar_arrive_expect_tx(&bars->v_full[vs], (uint32_t)C::kTileBytes);
          ptx::tma_load_3d_pair(dst, &tmV, ptx::map_cluster(ptx::smem_addr(&bars->v_full[vs]), 0), (int)crank * 64, j0,
                                b * a.Hkv + hk);
          ++issued[vs];
          continue;
        }
        ptx::mbar_arrive_expect_tx(&bars->v_full[vs], (uint32_t)C::kTileBytes);
        for (int db = 0; db < C::kDB; ++db) {
          if (mc)
            ptx::tma_load_3d_mc(dst + db * C::kKVBlock + crank * (kBN2 / 2) * 128, &tmV, &bars->v_full[vs], db * 64,
                                j0 + (int)crank * (kBN2 / 2), b * a.Hkv + hk, kPairMask);
          else
            ptx::tma_load_3d(dst + db * C::kKVBlock, &tmV, &bars->v_full[vs], db * 64, j0, b * a.Hkv + hk);
        }
        ++issued[vs];
      }
      for (int s = 0; s < kPair2Slots; ++s)
        if (issued[s])
          ptx::mbar_wait(kPair ? &bars->v_empty[s] : &bars->v_full[s], (issued[s] - 1) & 1, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1 || warp == kP2Threads / 32 - 1) {
    // ------------------------------------------------------------------ S issuer of tile x
    // one issuing thread per row tile: the short (N = 64) S products of the two tiles are
    // issued in parallel
    const int x = warp == 1 ? 0 : 1;
    if (lane == 0 && issuer_cta) {
      if (nts > 0 && ptx::mbar_wait(&bars->q_full, 0, abort_flag)) {
        constexpr uint32_t idS = ptx::idesc_bf16(kPair ? 2 * kRows : kRows, kBN2, false, false);
        const uint32_t qaddr = ptx::smem_addr(sQ + x * C::kQTile);
        uint64_t adq[8];  // the Q tile's A descriptors, one per 16-element K step
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          adq[kk] = ptx::sdesc_sw128(qaddr + (kk >> 2) * C::kQBlock + (kk & 3) * 32, 16, 1024);
        for (int t = 0; t < nts; ++t) {
          const int ks = t % kPair2Slots, buf = t & 1;
          if (!ptx::mbar_wait(&bars->k_full[ks], (t / kPair2Slots) & 1, abort_flag)) break;
          if (t < ntx[x]) {
            // S_X(t) overwrites P_X(t - 2) in this buffer: wait for PV_X(t - 2)
            if (t >= 2 && !ptx::mbar_wait(&bars->pv_done[x][buf], ((t - 2) >> 1) & 1, abort_flag)) break;
            ptx::tc_fence_after();
            const uint32_t kaddr = ptx::smem_addr(sK + ks * C::kTileBytes);
            if constexpr (!kPair && D == 128) {
              s_product_d128(tmem + x * kRows + buf * kBN2, adq, ptx::sdesc_sw128(kaddr, 16, 1024), idS);
            } else
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;  // 16-element K step inside a 128-byte row
              const uint64_t ad = ptx::sdesc_sw128(qaddr + (kk >> 2) * C::kQBlock + off, 16, 1024);
              if constexpr (kPair) {  // 32 keys per CTA: column blocks of 4 KB
                const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * (C::kKVBlock / 2) + off, 16, 1024);
                ptx::mma_bf16_ss_pair(tmem + x * kRows + buf * kBN2, ad, bd, idS, kk > 0 ? 1u : 0u);
              } else {
                const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * C::kKVBlock + off, 16, 1024);
                ptx::mma_bf16_ss(tmem + x * kRows + buf * kBN2, ad, bd, idS, kk > 0 ? 1u : 0u);
              }
            }
            if constexpr (kPair)
              ptx::mma_commit_pair_mc(&bars->s_full[x][buf], kPairMask);
            else
              ptx::mma_commit(&bars->s_full[x][buf]);
          }
          if constexpr (kPair)
            ptx::mma_commit_pair_mc(&bars->k_empty[ks], kPairMask);
          else if (mc)  // this tile is done with the K slot (in both CTAs' rings)
            ptx::mma_commit_mc(&bars->k_empty[ks], kPairMask);
          else
            ptx::mma_commit(&bars->k_empty[ks]);
        }
      }
      if constexpr (kPair)
        ptx::mma_commit_pair(&bars->s_done[x]);
      else
        ptx::mma_commit(&bars->s_done[x]);
      ptx::mbar_wait(&bars->s_done[x], 0, abort_flag);
    }
    __syncwarp();
  } else if (warp == kP2Threads / 32 - 2) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0 && issuer_cta) {
      constexpr uint32_t idO = ptx::idesc_bf16(kPair ? 2 * kRows : kRows, D, false, true);
      bool ok = true;
      for (int t = 0; ok && t < nts; ++t) {
        const int vs = t % kPair2Slots, buf = t & 1;
        if (!ptx::mbar_wait(&bars->v_full[vs], (t / kPair2Slots) & 1, abort_flag)) break;
        const uint32_t vaddr = ptx::smem_addr(sV + vs * C::kTileBytes);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (t >= ntx[x]) continue;
          if (!(kPair ? ptx::mbar_wait_cluster(&bars->p_full[x][buf], (t >> 1) & 1, abort_flag)
                      : ptx::mbar_wait(&bars->p_full[x][buf], (t >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t pcol = tmem + x * kRows + buf * kBN2;  // P: 8 columns per 16 keys
          if constexpr (!kPair && D == 128) {
            pv_product_d128(tmem + C::kColO + x * kRows, pcol, ptx::sdesc_sw128(vaddr, C::kKVBlock, 1024), idO,
                            t > 0 ? 1u : 0u);
          } else
#pragma unroll
          for (int kk = 0; kk < kBN2 / 16; ++kk) {
            const uint64_t bd = ptx::sdesc_sw128(vaddr + kk * 16 * 128, C::kKVBlock, 1024);
            if constexpr (kPair)  // this CTA's 64 value columns of the 128
              ptx::mma_bf16_ts_pair(tmem + C::kColO + x * kRows, pcol + kk * 8, bd, idO, (t > 0 || kk > 0) ? 1u : 0u);
            else
              ptx::mma_bf16_ts(tmem + C::kColO + x * kRows, pcol + kk * 8, bd, idO, (t > 0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (kPair)
            ptx::mma_commit_pair_mc(&bars->pv_done[x][buf], kPairMask);
          else
            ptx::mma_commit(&bars->pv_done[x][buf]);
        }
        if (ok) {
          if constexpr (kPair)
            ptx::mma_commit_pair_mc(&bars->v_empty[vs], kPairMask);
          else if (mc)
            ptx::mma_commit_mc(&bars->v_empty[vs], kPairMask);
          else
            ptx::mma_commit(&bars->v_empty[vs]);
        }
      }
      if constexpr (kPair)
        ptx::mma_commit_pair_mc(&bars->o_done, kPairMask);
      else
        ptx::mma_commit(&bars->o_done);
      ptx::mbar_wait(&bars->o_done, 0, abort_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax rows
    const int x = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int g = r / a.NT, il = r % a.NT;
    const int node = i0[x] + il;
    const bool valid = (g < a.G) && (node < a.N) && (r < rows_used) && !(node > 0 && s_par[node] == -1);
    const int mnode = valid ? node : 0;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t colS = tmem + lane_base + x * kRows;
    const uint32_t colO = tmem + lane_base + C::kColO + x * kRows;
    const int ntm = ntx[x];
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntm; ++t) {
      const int buf = t & 1;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->s_full[x][buf], (t >> 1) & 1, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      const int j0 = (t_begin + t) * kBN2;
      const uint64_t vis = key_mask(j0, a.P, a.N, mnode, s_par);
      float sv[64];
      ptx::tmem_ld32(colS + buf * kBN2, sv);
      ptx::tmem_ld32(colS + buf * kBN2 + 32, sv + 32);
      ptx::tmem_wait_ld();
      if (vis != ~0ull) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (!((vis >> j) & 1ull)) sv[j] = -INFINITY;
      }
      // P = 2^(S c - m_run) against the running reference m_run, which moves (and O is
      // rescaled) only when a score exceeds it by more than 2^8.  Such a score makes its P
      // exceed 2^8 and so the tile's sum of P reach 2^8: the row maximum is taken only for
      // those tiles (and for the first tile with a visible key), and a moved reference
      // redoes the exponentials.  The decisions are those of taking the maximum of every
      // tile first, up to rounding of a score within an ulp of the 2^8 boundary (either
      // choice gives the same softmax).
      float alpha = 1.f;
      bool need = false;
      bool checked = false;
      if (m_run == -INFINITY) {
        m_run = max64(sv, -INFINITY) * a.c;  // stays -inf while no key is visible
        checked = true;
      }
      uint32_t pw[32];
      float lsum;
      for (;;) {
        lsum = exp_p64(sv, a.c, m_run, pw);
        if (checked || lsum < kRescaleSum) break;
        checked = true;
        const float tms = max64(sv, -INFINITY) * a.c;
        if (!(tms > m_run + kRescaleLog2)) break;
        alpha = ptx::ex2(m_run - tms);
        need = true;
        m_run = tms;
      }
      ptx::tmem_st32u(colS + buf * kBN2, pw);  // P over the first half of this S buffer
      if (__any_sync(0xffffffffu, need) && t > 0) {
        // O_X must hold all of PV_X(t - 1) before it is rescaled (S_X(t) may have been
        // computed while PV_X(t - 1) was still running); PV_X(t) waits for P_X(t)
        ok = __all_sync(0xffffffffu,
                        ptx::mbar_wait(&bars->pv_done[x][(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float ov[32];
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] *= alpha;
          ptx::tmem_st32(colO + c0, ov);
        }
      }
      l_run = l_run * alpha + lsum;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // SM pair: the odd CTA's warps arrive on the even (issuing) CTA's barrier; P is in
        // TMEM, ordered by the tcgen05 wait and fence above, so no release is needed
        if (kPair && crank != 0)
          ptx::mbar_arrive_cluster_relaxed(ptx::map_cluster(ptx::smem_addr(&bars->p_full[x][buf]), 0));
        else
          ptx::mbar_arrive(&bars->p_full[x][buf]);
      }
    }
    // ---- epilogue (as in attn_pair_kernel): every MMA is complete at o_done
    bool have_o = false;
    if (nt > 0) {
      const bool done = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->o_done, 0, abort_flag));
      have_o = done && ok && ntm > 0;
      if (done) ptx::tc_fence_after();
    }
    const int hh = hk * a.G + g;
    const size_t orow = (((size_t)b * a.Hq + hh) * a.N + node) * D;
    if (a.splits == 1) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = ptx::cvt_bf16x2(ov[8 * k + 0] * inv, ov[8 * k + 1] * inv);
            u.y = ptx::cvt_bf16x2(ov[8 * k + 2] * inv, ov[8 * k + 3] * inv);
            u.z = ptx::cvt_bf16x2(ov[8 * k + 4] * inv, ov[8 * k + 5] * inv);
            u.w = ptx::cvt_bf16x2(ov[8 * k + 6] * inv, ov[8 * k + 7] * inv);
            dst[k] = u;
          }
        }
      }
    } else {
      const int R = x * kRows + r;
      unsigned char* part = sK;
      float2* ml = reinterpret_cast<float2*>(sQ);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int chunk = c0 / 4 + k;
          *reinterpret_cast<float4*>(part + (size_t)R * D * 4 + ((chunk ^ (R & 7)) << 4)) =
              make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
        }
      }
      ml[R] = make_float2(have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
    }
    ptx::tc_fence_before();
  }
  __syncwarp();
  if (a.splits > 1) {
    ptx::cluster_sync();
    {
      const int S = a.splits;
      constexpr int kPRows = 2 * kRows;
      const int R = (kPRows + S - 1) / S;
      const int r0 = split * R, r1 = min(kPRows, r0 + R);
      const int nrows = max(0, r1 - r0);
      constexpr int kChunks = D / 4;
      const uint32_t part_local = ptx::smem_addr(sK);
      const uint32_t ml_local = ptx::smem_addr(sQ);
      for (int item = threadIdx.x; item < nrows * kChunks; item += kP2Threads) {
        const int rr = r0 + item / kChunks;
        const int ch = item % kChunks;
        const int xx = rr >= kRows ? 1 : 0, rt = rr - xx * kRows;
        const int gg = rt / a.NT, ii = i0[xx] + rt % a.NT;
        if (gg >= a.G || ii >= a.N || rt >= rows_used || (ii > 0 && s_par[ii] == -1)) continue;
        float2 mlv[kMaxSplits];
        float4 xv[kMaxSplits];
        const uint32_t moff = (uint32_t)(rr * 8);
        const uint32_t xoff = (uint32_t)(rr * D * 4 + ((ch ^ (rr & 7)) << 4));
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S) {
            mlv[s2] = ptx::ld_cluster_f32x2(ptx::map_cluster(ml_local, s2) + moff);
            xv[s2] = ptx::ld_cluster_f32x4(ptx::map_cluster(part_local, s2) + xoff);
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2)
          if (s2 < S) M = fmaxf(M, mlv[s2].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s2 = 0; s2 < kMaxSplits; ++s2) {
          if (s2 < S && mlv[s2].x != -INFINITY) {
            const float w = ptx::ex2(mlv[s2].x - M);
            L = fmaf(mlv[s2].y, w, L);
            acc.x = fmaf(w, xv[s2].x, acc.x);
            acc.y = fmaf(w, xv[s2].y, acc.y);
            acc.z = fmaf(w, xv[s2].z, acc.z);
            acc.w = fmaf(w, xv[s2].w, acc.w);
          }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t o2 = (((size_t)b * a.Hq + hk * a.G + gg) * a.N + ii) * D + ch * 4;
        uint2 u;
        u.x = ptx::cvt_bf16x2(acc.x * inv, acc.y * inv);
        u.y = ptx::cvt_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + o2) = u;
      }
    }
    __syncwarp();
    ptx::cluster_sync();
  }
  __syncthreads();
  // the peer's multicasts and commit arrivals into this CTA are done (SM pair: and the
  // pair's MMAs, which read and write both CTAs)
  if (mc || kPair) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (kPair)
      ptx::tmem_dealloc_pair(tmem, C::kTmemCols);
    else
      ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// attn_stream_kernel: the paired 64-key pipeline of attn_pair2_kernel (in its earlier form,
// one S issuing thread for both row tiles) under a persistent schedule.  The work of a launch is the list of all (tile pair, 64-key KV tile) steps,
// unit by unit (a unit = one tile pair of one (sequence, KV head)); every CTA of the
// grid (one per SM of its share) takes an equal contiguous range of it, so that 128
// units on 152 SMs keep every SM busy instead of leaving 24 idle.  A range covers whole
// units and at most one partial unit at each end.  A partial unit's pieces write their
// unnormalised O and (m, l) rows to the workspace; one acquire-release atomic per unit
// counts them and the CTA that adds the last piece merges the rows and writes the output
// (no CTA ever waits for another).  Per piece, the Q tiles are reloaded once the S
// products of the previous piece are done (q_empty), and the first PV product of a piece
// waits until the softmax warps have read the previous piece's O (o_free).
constexpr int kMaxMP = 64;      // tile pairs per (sequence, KV head): N = 1024 rows at G = 16
constexpr int kMaxPieces = 8;   // units one persistent CTA may touch (the plan keeps below it)

struct StreamArgs {
  long long W;          // 64-key steps of the whole launch
  int C;                // CTAs
  int MP;               // tile pairs per (sequence, KV head)
  int Tg;               // steps per (sequence, KV head) = pre[MP]
  int pre[kMaxMP + 1];  // prefix sums of the tile pairs' step counts
  float* ws_o;          // [2C][256][D] unnormalised partial O rows
  float2* ws_ml;        // [2C][256] (running max in log2 units, sum)
  unsigned* cnt;        // [B * Hkv * MP] pieces of each unit finished
};

struct StreamPiece {
  int g, mp, ta, tb;  // unit (g = sequence * Hkv + KV head, tile pair mp), steps [ta, tb)
  int slot;           // workspace slot of a partial piece; -1 when the piece is its whole unit
};

struct StreamBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kPair2Slots];
  uint64_t k_empty[kPair2Slots];
  uint64_t v_full[kPair2Slots];
  uint64_t v_empty[kPair2Slots];
  uint64_t s_full[2][2];
  uint64_t p_full[2][2];
  uint64_t pv_done[2][2];
  uint64_t o_done, o_free, s_done;
  uint32_t tmem_base;
  int abort;
  int npiece;
  int last;  // this CTA adds the last piece of the current unit
  StreamPiece piece[kMaxPieces];
};

// the CTA whose range holds step w: the largest c with floor(c W / C) <= w
__device__ __forceinline__ int stream_owner(long long w, const StreamArgs& s) {
  return (int)((w * s.C + s.C - 1) / s.W);
}
__device__ __forceinline__ long long stream_start(int c, const StreamArgs& s) { return (long long)c * s.W / s.C; }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_stream_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, TcArgs a, const __grid_constant__ StreamArgs sa) {
  ptx::griddep_launch_dependents();
  using C = Pair2Cfg<D>;
  static_assert(sizeof(StreamBars) <= 512, "stream barriers fit the barrier region");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t mis = ptx::smem_addr(smem_raw) & 1023u;
  unsigned char* sm = smem_raw + ((1024u - mis) & 1023u);
  unsigned char* sQ = sm + C::kOffQ;
  unsigned char* sK = sm + C::kOffK;
  unsigned char* sV = sm + C::kOffV;
  int* s_par = reinterpret_cast<int*>(sm + C::kOffPar);
  StreamBars* bars = reinterpret_cast<StreamBars*>(sm + C::kOffBar);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int rows_used = a.G * a.NT;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 1);
    ptx::mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kPair2Slots; ++s) {
      ptx::mbar_init(&bars->k_full[s], 1);
      ptx::mbar_init(&bars->k_empty[s], 1);
      ptx::mbar_init(&bars->v_full[s], 1);
      ptx::mbar_init(&bars->v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x)
      for (int u = 0; u < 2; ++u) {
        ptx::mbar_init(&bars->s_full[x][u], 1);
        ptx::mbar_init(&bars->p_full[x][u], 4);
        ptx::mbar_init(&bars->pv_done[x][u], 1);
      }
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->o_free, 8);
    ptx::mbar_init(&bars->s_done, 1);
    bars->abort = 0;
    // this CTA's pieces: its range [start(c), start(c + 1)) cut at unit boundaries
    const long long w0 = stream_start(cta, sa), w1 = stream_start(cta + 1, sa);
    int np = 0;
    for (long long w = w0; w < w1 && np < kMaxPieces; ++np) {
      const int g = (int)(w / sa.Tg);
      const int rr = (int)(w - (long long)g * sa.Tg);
      int mp = 0;
      while (sa.pre[mp + 1] <= rr) ++mp;
      const int tmp = sa.pre[mp + 1] - sa.pre[mp];
      const int ta = rr - sa.pre[mp];
      const int tb = (int)min((long long)tmp, ta + (w1 - w));
      StreamPiece pc{g, mp, ta, tb, -1};
      if (ta > 0 || tb < tmp) pc.slot = 2 * cta + (w > w0 ? 1 : 0);  // first or last piece of the range
      bars->piece[np] = pc;
      w += tb - ta;
    }
    bars->npiece = np;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {  // kernel parameters: safe before the wait
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  // the set-up above touches only shared memory, TMEM and parameters, so it overlaps the
  // previous kernel's tail (programmatic dependent launch); global memory after this
  ptx::griddep_wait();
  if (warp >= 2) {
    // zero the Q rows that no TMA box fills (the same rows in every unit)
    const int t = threadIdx.x - 64;
    for (int r = rows_used + t; r < 2 * kRows; r += kThreads - 64) {
      const int x = r >= kRows ? 1 : 0, rr = r - x * kRows;
      if (rr < rows_used) continue;
      for (int db = 0; db < C::kDB; ++db) {
        uint4* row = reinterpret_cast<uint4*>(sQ + x * C::kQTile + db * C::kQBlock + rr * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) row[k] = make_uint4(0, 0, 0, 0);
      }
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int np = bars->npiece;

  // per-piece geometry, identical in every role
  auto geom = [&](const StreamPiece& pc, int* i0, int* ntx) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      i0[x] = (2 * pc.mp + x) * a.NT;
      const int tall = i0[x] < a.N ? (a.P + min(a.N, i0[x] + a.NT) + kBN2 - 1) / kBN2 : 0;
      ntx[x] = max(0, min(tall, pc.tb) - pc.ta);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producers
    if (lane == 0) {
      int issued[kPair2Slots] = {0, 0, 0, 0};
      long long gk = 0;
      for (int p = 0; p < np && !*abort_flag; ++p) {
        const StreamPiece pc = bars->piece[p];
        int i0[2], ntx[2];
        geom(pc, i0, ntx);
        const int b = pc.g / a.Hkv, hk = pc.g % a.Hkv;
        const int nt = max(ntx[0], ntx[1]);
        // Q of this unit once the S products of the previous piece are done
        if (p > 0 && !ptx::mbar_wait(&bars->q_empty, (p - 1) & 1, abort_flag)) break;
        uint32_t qbytes = 0;
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (ntx[x] > 0) qbytes += (uint32_t)(rows_used * 128 * C::kDB);
        ptx::mbar_arrive_expect_tx(&bars->q_full, qbytes);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (ntx[x] > 0)
            for (int g = 0; g < a.G; ++g)
              for (int db = 0; db < C::kDB; ++db)
                ptx::tma_load_3d(sQ + x * C::kQTile + db * C::kQBlock + g * a.NT * 128, &tmQ, &bars->q_full,
                                 db * 64, i0[x], b * a.Hq + hk * a.G + g);
        for (int t = 0; t < nt; ++t, ++gk) {
          const int ks = (int)(gk % kPair2Slots);
          if (gk >= kPair2Slots &&
              !ptx::mbar_wait(&bars->k_empty[ks], (uint32_t)((gk / kPair2Slots) - 1) & 1, abort_flag))
            break;
          unsigned char* dst = sK + ks * C::kTileBytes;
          ptx::mbar_arrive_expect_tx(&bars->k_full[ks], (uint32_t)C::kTileBytes);
          for (int db = 0; db < C::kDB; ++db)
            ptx::tma_load_3d(dst + db * C::kKVBlock, &tmK, &bars->k_full[ks], db * 64, (pc.ta + t) * kBN2,
                             b * a.Hkv + hk);
          ++issued[ks];
        }
      }
      if (np > 0) ptx::mbar_wait(&bars->q_full, (np - 1) & 1, abort_flag);
      for (int s = 0; s < kPair2Slots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->k_full[s], (issued[s] - 1) & 1, abort_flag);
    } else if (lane == 1) {
      int issued[kPair2Slots] = {0, 0, 0, 0};
      long long gv = 0;
      for (int p = 0; p < np && !*abort_flag; ++p) {
        const StreamPiece pc = bars->piece[p];
        int i0[2], ntx[2];
        geom(pc, i0, ntx);
        const int b = pc.g / a.Hkv, hk = pc.g % a.Hkv;
        const int nt = max(ntx[0], ntx[1]);
        for (int t = 0; t < nt; ++t, ++gv) {
          const int vs = (int)(gv % kPair2Slots);
          if (gv >= kPair2Slots &&
              !ptx::mbar_wait(&bars->v_empty[vs], (uint32_t)((gv / kPair2Slots) - 1) & 1, abort_flag))
            break;
          unsigned char* dst = sV + vs * C::kTileBytes;
          ptx::mbar_arrive_expect_tx(&bars->v_full[vs], (uint32_t)C::kTileBytes);
          for (int db = 0; db < C::kDB; ++db)
            ptx::tma_load_3d(dst + db * C::kKVBlock, &tmV, &bars->v_full[vs], db * 64, (pc.ta + t) * kBN2,
                             b * a.Hkv + hk);
          ++issued[vs];
        }
      }
      for (int s = 0; s < kPair2Slots; ++s)
        if (issued[s]) ptx::mbar_wait(&bars->v_full[s], (issued[s] - 1) & 1, abort_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t idS = ptx::idesc_bf16(kRows, kBN2, false, false);
      long long gk = 0;
      int cs[2] = {0, 0};  // S products issued so far per row tile (buffer = cs & 1)
      bool ok = true;
      for (int p = 0; ok && p < np; ++p) {
        const StreamPiece pc = bars->piece[p];
        int i0[2], ntx[2];
        geom(pc, i0, ntx);
        const int nt = max(ntx[0], ntx[1]);
        if (!ptx::mbar_wait(&bars->q_full, p & 1, abort_flag)) break;
        for (int t = 0; ok && t < nt; ++t, ++gk) {
          const int ks = (int)(gk % kPair2Slots);
          if (!ptx::mbar_wait(&bars->k_full[ks], (uint32_t)(gk / kPair2Slots) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t kaddr = ptx::smem_addr(sK + ks * C::kTileBytes);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (t >= ntx[x]) continue;
            const int buf = cs[x] & 1;
            // S overwrites the P of two products back in this buffer: wait for its PV
            if (cs[x] >= 2 && !ptx::mbar_wait(&bars->pv_done[x][buf], ((cs[x] - 2) >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t qaddr = ptx::smem_addr(sQ + x * C::kQTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk & 3) * 32;
              const uint64_t ad = ptx::sdesc_sw128(qaddr + (kk >> 2) * C::kQBlock + off, 16, 1024);
              const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * C::kKVBlock + off, 16, 1024);
              ptx::mma_bf16_ss(tmem + x * kRows + buf * kBN2, ad, bd, idS, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(&bars->s_full[x][buf]);
            ++cs[x];
          }
          if (ok) ptx::mma_commit(&bars->k_empty[ks]);
        }
        if (ok) ptx::mma_commit(&bars->q_empty);  // the Q tiles are free once these S products are done
      }
      ptx::mma_commit(&bars->s_done);
      ptx::mbar_wait(&bars->s_done, 0, abort_flag);
    }
    __syncwarp();
  } else if (warp == kThreads / 32 - 1) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t idO = ptx::idesc_bf16(kRows, D, false, true);
      long long gv = 0;
      int cp[2] = {0, 0};
      bool ok = true;
      for (int p = 0; ok && p < np; ++p) {
        const StreamPiece pc = bars->piece[p];
        int i0[2], ntx[2];
        geom(pc, i0, ntx);
        const int nt = max(ntx[0], ntx[1]);
        // the first PV of a piece overwrites O: the softmax warps have read the last one
        if (p > 0 && !ptx::mbar_wait(&bars->o_free, (p - 1) & 1, abort_flag)) break;
        for (int t = 0; ok && t < nt; ++t, ++gv) {
          const int vs = (int)(gv % kPair2Slots);
          if (!ptx::mbar_wait(&bars->v_full[vs], (uint32_t)(gv / kPair2Slots) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t vaddr = ptx::smem_addr(sV + vs * C::kTileBytes);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (t >= ntx[x]) continue;
            const int buf = cp[x] & 1;
            if (!ptx::mbar_wait(&bars->p_full[x][buf], (cp[x] >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t pcol = tmem + x * kRows + buf * kBN2;
#pragma unroll
            for (int kk = 0; kk < kBN2 / 16; ++kk) {
              const uint64_t bd = ptx::sdesc_sw128(vaddr + kk * 16 * 128, C::kKVBlock, 1024);
              ptx::mma_bf16_ts(tmem + C::kColO + x * kRows, pcol + kk * 8, bd, idO, (t > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(&bars->pv_done[x][buf]);
            ++cp[x];
          }
          if (ok) ptx::mma_commit(&bars->v_empty[vs]);
        }
        ptx::mma_commit(&bars->o_done);  // every product of this piece (phase p)
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax rows
    const int x = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int R = x * kRows + r;  // row of the pair (workspace row)
    const int g = r / a.NT, il = r % a.NT;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t colS = tmem + lane_base + x * kRows;
    const uint32_t colO = tmem + lane_base + C::kColO + x * kRows;
    const int st = threadIdx.x - 64;  // 0..255 over the softmax warps
    int cs = 0;
    int cur_b = -1;
    bool ok = true;
    for (int p = 0; p < np; ++p) {
      const StreamPiece pc = bars->piece[p];
      int i0[2], ntx[2];
      geom(pc, i0, ntx);
      const int b = pc.g / a.Hkv, hk = pc.g % a.Hkv;
      if (b != cur_b) {  // the parent array of this piece's sequence
        asm volatile("bar.sync 1, 256;" ::: "memory");
        int bad = 0;
        for (int c = st; c < a.N; c += 256) {
          const int pr = a.parent[(size_t)b * a.N + c];
          s_par[c] = pr;
          const bool prev_pad = c >= 2 && a.parent[(size_t)b * a.N + c - 1] == -1;
          if (!((c == 0) ? (pr == -1) : (pr == -1 || (pr >= 0 && pr < c && !prev_pad)))) bad = 1;
        }
        if (bad) set_dev_status(a.dev_status, TV_DEV_BAD_TREE);
        asm volatile("bar.sync 1, 256;" ::: "memory");
        cur_b = b;
      }
      const int node = i0[x] + il;
      const bool valid = (g < a.G) && (node < a.N) && (r < rows_used) && !(node > 0 && s_par[node] == -1);
      const int mnode = valid ? node : 0;
      const int ntm = ntx[x];
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; ok && t < ntm; ++t, ++cs) {
        const int buf = cs & 1;
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->s_full[x][buf], (cs >> 1) & 1, abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
        const uint64_t vis = key_mask((pc.ta + t) * kBN2, a.P, a.N, mnode, s_par);
        float sv[64];
        ptx::tmem_ld32(colS + buf * kBN2, sv);
        ptx::tmem_ld32(colS + buf * kBN2 + 32, sv + 32);
        ptx::tmem_wait_ld();
        if (vis != ~0ull) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (!((vis >> j) & 1ull)) sv[j] = -INFINITY;
        }
        const float tms = max64(sv, -INFINITY) * a.c;
        float alpha = 1.f;
        bool need = false;
        if (tms > m_run + kRescaleLog2) {
          if (m_run != -INFINITY) {
            alpha = ptx::ex2(m_run - tms);
            need = true;
          }
          m_run = tms;
        }
        uint32_t pw[32];
        const float lsum = exp_p64(sv, a.c, m_run, pw);
        ptx::tmem_st32u(colS + buf * kBN2, pw);
        if (__any_sync(0xffffffffu, need) && t > 0) {
          ok = __all_sync(0xffffffffu,
                          ptx::mbar_wait(&bars->pv_done[x][(cs - 1) & 1], ((cs - 1) >> 1) & 1, abort_flag));
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float ov[32];
            ptx::tmem_ld32(colO + c0, ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) ov[k] *= alpha;
            ptx::tmem_st32(colO + c0, ov);
          }
        }
        l_run = l_run * alpha + lsum;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->p_full[x][buf]);
      }
      // ---- epilogue of the piece: every product of it is complete at o_done (phase p)
      const bool done = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->o_done, p & 1, abort_flag));
      if (done) ptx::tc_fence_after();
      const bool have_o = done && ok && ntm > 0;
      const size_t orow = (((size_t)b * a.Hq + hk * a.G + g) * a.N + node) * D;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      float4* wrow = reinterpret_cast<float4*>(sa.ws_o + ((size_t)max(pc.slot, 0) * 2 * kRows + R) * D);
      // O in 32-column chunks: the output row (whole unit) or the parked partial row
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (have_o) {
          ptx::tmem_ld32(colO + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        }
        if (pc.slot >= 0) {
#pragma unroll
          for (int k = 0; k < 8; ++k) wrow[c0 / 4 + k] = make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = ptx::cvt_bf16x2(ov[8 * k + 0] * inv, ov[8 * k + 1] * inv);
            u.y = ptx::cvt_bf16x2(ov[8 * k + 2] * inv, ov[8 * k + 3] * inv);
            u.z = ptx::cvt_bf16x2(ov[8 * k + 4] * inv, ov[8 * k + 5] * inv);
            u.w = ptx::cvt_bf16x2(ov[8 * k + 6] * inv, ov[8 * k + 7] * inv);
            dst[k] = u;
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->o_free);  // O may be overwritten by the next piece
      if (pc.slot < 0) continue;
      // partial piece: count it; the CTA adding the last piece of the unit merges
      sa.ws_ml[(size_t)pc.slot * 2 * kRows + R] = make_float2(have_o ? m_run : -INFINITY, have_o ? l_run : 0.f);
      const int unit = pc.g * sa.MP + pc.mp;
      const long long U0 = (long long)pc.g * sa.Tg + sa.pre[pc.mp];
      const long long U1 = U0 + (sa.pre[pc.mp + 1] - sa.pre[pc.mp]);
      const int c_lo = stream_owner(U0, sa), c_hi = stream_owner(U1 - 1, sa);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (st == 0) {
        const unsigned prev = ptx::atom_add_acq_rel_gpu(sa.cnt + unit, 1u);
        bars->last = prev + 1 == (unsigned)(c_hi - c_lo + 1);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (!bars->last) continue;
      if (st == 0) sa.cnt[unit] = 0;  // ready for the next launch
      if (!valid) continue;
      // merge this row over the unit's pieces (CTAs c_lo..c_hi), 32 columns at a time
      float M = -INFINITY;
      for (int c = c_lo; c <= c_hi; ++c) {
        const int slot = 2 * c + ((c == c_lo && U0 > stream_start(c, sa)) ? 1 : 0);
        M = fmaxf(M, __ldcg(&sa.ws_ml[(size_t)slot * 2 * kRows + R]).x);
      }
      float L = 0.f;
      for (int c = c_lo; c <= c_hi; ++c) {
        const int slot = 2 * c + ((c == c_lo && U0 > stream_start(c, sa)) ? 1 : 0);
        const float2 ml = __ldcg(&sa.ws_ml[(size_t)slot * 2 * kRows + R]);
        if (ml.x != -INFINITY) L = fmaf(ml.y, ptx::ex2(ml.x - M), L);
      }
      const float minv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) ov[k] = 0.f;
        for (int c = c_lo; c <= c_hi; ++c) {
          const int slot = 2 * c + ((c == c_lo && U0 > stream_start(c, sa)) ? 1 : 0);
          const float2 ml = __ldcg(&sa.ws_ml[(size_t)slot * 2 * kRows + R]);
          if (ml.x == -INFINITY) continue;
          const float w = ptx::ex2(ml.x - M);
          const float4* src = reinterpret_cast<const float4*>(sa.ws_o + ((size_t)slot * 2 * kRows + R) * D + c0);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 v = __ldcg(src + k);
            ov[4 * k] = fmaf(w, v.x, ov[4 * k]);
            ov[4 * k + 1] = fmaf(w, v.y, ov[4 * k + 1]);
            ov[4 * k + 2] = fmaf(w, v.z, ov[4 * k + 2]);
            ov[4 * k + 3] = fmaf(w, v.w, ov[4 * k + 3]);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + orow + c0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 u;
          u.x = ptx::cvt_bf16x2(ov[8 * k + 0] * minv, ov[8 * k + 1] * minv);
          u.y = ptx::cvt_bf16x2(ov[8 * k + 2] * minv, ov[8 * k + 3] * minv);
          u.z = ptx::cvt_bf16x2(ov[8 * k + 4] * minv, ov[8 * k + 5] * minv);
          u.w = ptx::cvt_bf16x2(ov[8 * k + 6] * minv, ov[8 * k + 7] * minv);
          dst[k] = u;
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && bars->abort) set_dev_status(a.dev_status, TV_DEV_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D bf16 map {D, rows, planes} with a 64 x box_rows x 1 box, 128-byte swizzle.
static bool encode_3d(CUtensorMap* m, const void* base, int D, int rows, long long planes, long long row_stride_elems,
                      long long plane_stride_elems, int box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride_elems * 2, (cuuint64_t)plane_stride_elems * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int device_sms() {
  static std::atomic<int> cache[64];  // 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Work geometry of the persistent schedule: per tile pair mp of a (sequence, KV head), its
// 64-key step count max over its two row tiles of ceil((P + last node + 1) / 64); prefix
// sums in sa->pre.  Returns false when the shape has more tile pairs than the kernel
// takes.  *tmin: the smallest unit.
static bool stream_geometry(int B, int Hkv, int NT, int mtiles, int P, int N, StreamArgs* sa, int* tmin) {
  const int MP = (mtiles + 1) / 2;
  if (MP < 1 || MP > kMaxMP) return false;
  sa->MP = MP;
  sa->pre[0] = 0;
  int lo = 1 << 30;
  for (int mp = 0; mp < MP; ++mp) {
    int tu = 0;
    for (int x = 0; x < 2; ++x) {
      const int i0 = (2 * mp + x) * NT;
      if (i0 < N) tu = std::max(tu, (P + std::min(N, i0 + NT) + kBN2 - 1) / kBN2);
    }
    sa->pre[mp + 1] = sa->pre[mp] + tu;
    lo = std::min(lo, tu);
  }
  sa->Tg = sa->pre[MP];
  sa->W = (long long)B * Hkv * sa->Tg;
  *tmin = lo;
  return true;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// workspace of the persistent schedule on C CTAs: two partial slots per CTA (its first
// and last piece) of 256 rows x D fp32 plus (m, l), and one counter per unit
static size_t stream_ws_bytes(int C, int D, long long units) {
  return align256((size_t)2 * C * 2 * kRows * D * 4) + align256((size_t)2 * C * 2 * kRows * 8) +
         align256((size_t)units * 4);
}

// Kernel variants: 1 attn_tc_kernel (one 128-row tile per CTA, 128-key KV tiles),
// 2 attn_pair_kernel (two row tiles, 128-key KV tiles), 3 attn_pair2_kernel (two row
// tiles, 64-key KV tiles, two S buffers per row tile), 4 attn_stream_kernel (variant 3's
// pipeline on a persistent grid, equal work per SM), 5 attn_pair2_kernel on SM pairs
// (variant 3 with every product an M = 256 MMA over two CTAs' row tiles; D = 128).
template <int D, int kVar>
static const void* tc_kernel_fn() {
  if constexpr (kVar == 1) return reinterpret_cast<const void*>(attn_tc_kernel<D>);
  else if constexpr (kVar == 2) return reinterpret_cast<const void*>(attn_pair_kernel<D>);
  else if constexpr (kVar == 3) return reinterpret_cast<const void*>(attn_pair2_kernel<D, false>);
  else if constexpr (kVar == 5) return reinterpret_cast<const void*>(attn_pair2_kernel<D, true>);
  else return reinterpret_cast<const void*>(attn_stream_kernel<D>);
}
template <int D, int kVar>
static constexpr int tc_smem() {
  return kVar == 1 ? TcCfg<D>::kSmemAlloc : kVar == 2 ? PairCfg<D>::kSmemAlloc : Pair2Cfg<D>::kSmemAlloc;
}
constexpr int tc_threads(int var) { return var == 3 || var == 5 ? kP2Threads : kThreads; }
constexpr int tc_keys(int var) { return var >= 3 ? kBN2 : kBN; }  // keys per KV tile

// How many clusters of `s` CTAs of variant kVar can be resident at once on the current
// device (cached per device, variant and s).
template <int D, int kVar>
static int max_active_clusters(int s) {
  // one table per template instance: 0 = not queried yet, else the count + 1; threads that
  // query at the same time store the same value
  static std::atomic<int> cache[64][kMaxSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || s < 1 || s > kMaxSplits) return 0;
  const int known = cache[dev][s].load(std::memory_order_relaxed);
  if (known > 0) return known - 1;
  const void* fn = tc_kernel_fn<D, kVar>();
  const int smem = tc_smem<D, kVar>();
  int n = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s * 64, 1, 1);
    cfg.blockDim = dim3(tc_threads(kVar), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)s;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
  }
  cache[dev][s].store(n + 1, std::memory_order_relaxed);
  return n;
}

// Launch plan: kernel variant and KV splits minimising a wave model of the run time,
// (waves of clusters) x (KV tiles per CTA + a fixed per-CTA cost + the cluster merge when
// split) x (tile cost), in units of one 128-row x 128-key tile of attn_tc_kernel.  The
// constants are fitted to GB300 measurements over the qwen3 layer, sampling,
// long-context and budget-sweep shapes (every split count of both kernels): a CTA's
// set-up, pipeline fill and epilogue cost about 6 tiles, a cluster merge about 4.4, and
// 128 keys of a tile pair about 1.85 single tiles for attn_pair_kernel and 1.55 for
// attn_pair2_kernel (1.50-1.59 over the long-context, sampling and budget-sweep shapes).
constexpr double kFixedTiles = 6.0;
constexpr double kMergeTiles = 4.4;
constexpr double kPairTileCost = 1.85;
constexpr double kPair2TileCost = 1.55;

// SMs the attention may use (its share when one is set)
static int attention_sms() {
  const int nsm = device_sms();
  const int share = sm_share_attention();
  return share > 0 && share < nsm ? share : nsm;
}

template <int D, int kVar>
static double plan_cost(long long units, int t_all128, int s) {
  const int nsm = device_sms();
  int act = max_active_clusters<D, kVar>(s);
  if (act <= 0) return 1e300;
  const int use = attention_sms();
  if (use < nsm) act = std::max(1, (int)((long long)act * use / nsm));
  const long long waves = (units + act - 1) / act;
  const double tile = kVar == 1 ? 1.0 : kVar == 2 ? kPairTileCost : kPair2TileCost;
  return (double)waves * ((t_all128 + s - 1) / s + kFixedTiles + (s > 1 ? kMergeTiles : 0.0)) * tile;
}

// *var: 1, 2, 3 or 4 (see tc_kernel_fn).  The automatic choice considers variants 1 and
// 3: variant 3 was faster than variant 2 on every workload measured (3-8 % before it had
// one S issuer per row tile, 10-16 % since), and the
// persistent grid (4) slower than variant 3 on every one (3-6 % on long context, 28 % on
// sampling): these shapes run at the GB300's power limit, where 24 more busy SMs lower
// the SM clock instead of finishing sooner and the extra pieces and merges cost energy.
// 2 and 4 stay available when forced.  Variant 4 needs a workspace of
// stream_ws_bytes(C, ...) and a shape whose CTA ranges touch at most kMaxPieces units;
// *sa is filled when it is chosen.
template <int D>
static void choose_plan(int B, int Hkv, int NT, int mtiles, int P, int N, int* var, int* splits, StreamArgs* sa) {
  const int variant = attention_variant();
  const int forced = attention_splits();
  const int t_all128 = (P + N + kBN - 1) / kBN;
  const int fixed = variant >= 4 ? 3 : variant;  // variants 4 and 5 fall back to 3 where they cannot run
  double best_cost = 1e300;
  *var = 1;
  *splits = 1;
  for (int v = 1; v <= 3; ++v) {
    if (fixed != 0 && v != fixed) continue;
    if (variant == 0 && (v == 2 || (v == 3 && mtiles < 2))) continue;
    const long long units = (long long)B * Hkv * (v >= 2 ? (mtiles + 1) / 2 : mtiles);
    const int t_all = (P + N + tc_keys(v) - 1) / tc_keys(v);
    for (int s = 1; s <= kMaxSplits && s <= t_all; ++s) {
      if (forced > 0 && s != std::min(forced, t_all)) continue;
      const double c = v == 1   ? plan_cost<D, 1>(units, t_all128, s)
                       : v == 2 ? plan_cost<D, 2>(units, t_all128, s)
                                : plan_cost<D, 3>(units, t_all128, s);
      if (c < best_cost * 0.98) {  // prefer fewer splits and the single-tile kernel on near ties
        best_cost = c;
        *var = v;
        *splits = s;
      }
    }
  }
  if constexpr (D == 128) {
    // the SM-pair form (forced only): no KV splits, the tile pairs of a (sequence, KV
    // head) in twos.  It ties variant 3 on the long-context shape (402 us; 420 us in a
    // power-capped loop at a higher SM clock) and is 3-7 % slower on budget-sweep trees:
    // each SM's tensor pipe still runs 24 MMAs per 64-key step, the number that sets the
    // pace of variant 3
    const int pairs = (mtiles + 1) / 2;
    if (variant == 5 && forced <= 1 && pairs % 2 == 0 && max_active_clusters<D, 5>(1) > 0) {
      *var = 5;
      *splits = 1;
    }
  }
  if (variant == 4 && forced <= 1 && max_active_clusters<D, 3>(1) > 0) {
    StreamArgs g{};
    int tmin = 0;
    if (stream_geometry(B, Hkv, NT, mtiles, P, N, &g, &tmin) && tmin > 0) {
      const int C = (int)std::min<long long>(attention_sms(), g.W);
      const long long per = (g.W + C - 1) / C;  // steps per CTA
      // a range of `per` steps holds at most per / tmin whole units and a partial one at
      // each end
      if (per / tmin + 2 <= kMaxPieces) {
        *var = 4;
        *splits = 1;
        g.C = C;
        *sa = g;
      }
    }
  }
}

AttnPlan attn_plan(int B, int Hq, int Hkv, int D, int P, int N, tv_dtype dtype) {
  AttnPlan p{};
  const int G = Hkv > 0 ? Hq / Hkv : 0;
  p.tc = dtype == TV_BF16 && (D == 64 || D == 128) && G >= 1 && G <= 16 && (long long)G * N >= 64;
  if (!p.tc) return p;
  p.nt = (kRows / G) / 8 * 8;
  p.mtiles = (N + p.nt - 1) / p.nt;
  // the kernel variant and the KV splits are chosen at launch (choose_plan); split
  // partials stay in the cluster's shared memory, the persistent schedule's in the
  // workspace, sized for the whole device
  p.total = 0;
  int var = 1, spl = 1;
  StreamArgs sa{};
  if (D == 64)
    choose_plan<64>(B, Hkv, p.nt, p.mtiles, P, N, &var, &spl, &sa);
  else
    choose_plan<128>(B, Hkv, p.nt, p.mtiles, P, N, &var, &spl, &sa);
  if (var == 4) p.total = stream_ws_bytes(device_sms(), D, (long long)B * Hkv * sa.MP);
  return p;
}

template <int D, int kVar>
static cudaError_t launch_tc_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const TcArgs& a,
                               int B, int Hkv, cudaStream_t stream) {
  constexpr int smem = tc_smem<D, kVar>();
  cudaError_t e = cudaFuncSetAttribute(tc_kernel_fn<D, kVar>(), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int units = kVar >= 2 ? (a.MT + 1) / 2 : a.MT;  // CTAs per (b, kv head) and split
  const dim3 grid(units * a.splits, Hkv, B), block(tc_threads(kVar), 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  // SM pairs, K/V-sharing tile pairs, or KV splits
  attr[0].val.clusterDim.x = (kVar == 5 || a.mcast) ? 2u : (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if constexpr (kVar == 1)
    e = launch_pdl(attn_tc_kernel<D>, grid, block, smem, stream, attr, 1, mq, mk, mv, a);
  else if constexpr (kVar == 2)
    e = launch_pdl(attn_pair_kernel<D>, grid, block, smem, stream, attr, 1, mq, mk, mv, a);
  else if constexpr (kVar == 3)
    e = launch_pdl(attn_pair2_kernel<D, false>, grid, block, smem, stream, attr, 1, mq, mk, mv, a);
  else
    e = launch_pdl(attn_pair2_kernel<D, true>, grid, block, smem, stream, attr, 1, mq, mk, mv, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_stream_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                   const TcArgs& a, const StreamArgs& sa, cudaStream_t stream) {
  constexpr int smem = Pair2Cfg<D>::kSmemAlloc;
  cudaError_t e = cudaFuncSetAttribute(attn_stream_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the per-unit piece counters start at zero whatever an earlier (or aborted) call left
  const size_t units = (size_t)(sa.W / sa.Tg) * sa.MP;
  e = cudaMemsetAsync(sa.cnt, 0, units * sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_stream_kernel<D>, dim3((unsigned)sa.C), dim3(kThreads), smem, stream, nullptr, 0, mq, mk, mv, a,
                 sa);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

void attn_tc_choice(int B, int Hkv, int D, int P, int N, const AttnPlan& plan, int* var, int* splits) {
  StreamArgs sa{};
  if (D == 64)
    choose_plan<64>(B, Hkv, plan.nt, plan.mtiles, P, N, var, splits, &sa);
  else
    choose_plan<128>(B, Hkv, plan.nt, plan.mtiles, P, N, var, splits, &sa);
}

cudaError_t launch_attn_tc(const void* q, const void* k, const void* v, void* out, const int32_t* parent, int B,
                           int Hq, int Hkv, int D, int P, int N, int S, float scale, const AttnPlan& plan, char* ws,
                           size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  TcArgs a;
  a.out = out;
  a.parent = parent;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.P = P;
  a.G = Hq / Hkv;
  a.NT = plan.nt;
  a.MT = plan.mtiles;
  a.c = scale * kLog2e;
  a.dev_status = dev_status;
  a.mcast = 0;
  int var = 1;
  StreamArgs sa{};
  if (D == 64)
    choose_plan<64>(B, Hkv, plan.nt, plan.mtiles, P, N, &var, &a.splits, &sa);
  else
    choose_plan<128>(B, Hkv, plan.nt, plan.mtiles, P, N, &var, &a.splits, &sa);
  if (var == 4) {
    // the persistent schedule needs its partial slots; with a smaller workspace (one
    // sized under other settings) the unsplit paired kernel computes the same result
    const long long units = (long long)B * Hkv * sa.MP;
    if (!ws || ws_bytes < stream_ws_bytes(sa.C, D, units)) {
      var = 3;
      a.splits = 1;
    } else {
      sa.ws_o = reinterpret_cast<float*>(ws);
      sa.ws_ml = reinterpret_cast<float2*>(ws + align256((size_t)2 * sa.C * 2 * kRows * D * 4));
      sa.cnt = reinterpret_cast<unsigned*>(ws + align256((size_t)2 * sa.C * 2 * kRows * D * 4) +
                                           align256((size_t)2 * sa.C * 2 * kRows * 8));
    }
  }
  // the paired 64-key kernel without KV splits shares each K/V tile between the two tile
  // pairs of a cluster (each loads half of its rows, multicast to both) where the tile
  // pairs of a (sequence, KV head) come in twos and the prefix dominates the key range:
  // half the L2-to-SM traffic lowers power at the power limit (long-context attention
  // 427.7 -> 417.7 us in a long loop, SM clock 1905 -> 1972 MHz), while with short
  // prefixes the two CTAs' lockstep and the pair's extra tile cost more (budget-sweep
  // trees with P = 4 N: +2.5 %)
  const int pairs = (plan.mtiles + 1) / 2;
  a.mcast = (var == 3 && a.splits == 1 && pairs % 2 == 0 && (long long)P >= 64LL * N) ? 1 : 0;
  // rows of one K / V box: each CTA of an SM pair loads 32 keys of a K tile and all 64
  // keys of its half of a V tile
  const int kkeys = (var == 5 || a.mcast) ? kBN2 / 2 : tc_keys(var);
  const int vkeys = var == 5 ? kBN2 : kkeys;
  CUtensorMap mq, mk, mv;
  if (!encode_3d(&mq, q, D, N, (long long)B * Hq, D, (long long)N * D, plan.nt)) return cudaErrorInvalidValue;
  if (!encode_3d(&mk, k, D, P + N, (long long)B * Hkv, D, (long long)S * D, kkeys)) return cudaErrorInvalidValue;
  if (!encode_3d(&mv, v, D, P + N, (long long)B * Hkv, D, (long long)S * D, vkeys)) return cudaErrorInvalidValue;
  if (D == 64) {
    if (var == 1) return launch_tc_d<64, 1>(mq, mk, mv, a, B, Hkv, stream);
    if (var == 2) return launch_tc_d<64, 2>(mq, mk, mv, a, B, Hkv, stream);
    if (var == 4) return launch_stream_d<64>(mq, mk, mv, a, sa, stream);
    return launch_tc_d<64, 3>(mq, mk, mv, a, B, Hkv, stream);
  }
  if (var == 1) return launch_tc_d<128, 1>(mq, mk, mv, a, B, Hkv, stream);
  if (var == 2) return launch_tc_d<128, 2>(mq, mk, mv, a, B, Hkv, stream);
  if (var == 4) return launch_stream_d<128>(mq, mk, mv, a, sa, stream);
  if (var == 5) return launch_tc_d<128, 5>(mq, mk, mv, a, B, Hkv, stream);
  return launch_tc_d<128, 3>(mq, mk, mv, a, B, Hkv, stream);
}

}  // namespace tv
