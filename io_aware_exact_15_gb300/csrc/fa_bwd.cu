// Backward pass of exact attention by recomputation (FlashAttention hackmd
// summary, "Recomputation": the forward keeps only O and the softmax
// statistics; the backward rebuilds S and P block by block instead of
// reading an N x N matrix).  With lse from the forward and
// D_i = <dO_i, O_i> from the preprocess kernel, for each key tile j and every
// query tile i that reaches it:
//   S = Q_i K_j^T,  P = exp(scale*S - lse_i),  dP = dO_i V_j^T,
//   dS = P o (dP - D_i),
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i,  dQ_i += dS K_j  (dQ, dK scaled later).
//
// GB300 design (a unit = one key/value head x one 128-key tile; K_j, V_j
// stay in shared memory while the CTA walks the query tiles of every query
// head that reads this key/value head, so grouped K/V needs no atomics for
// dK and dV; persistent CTAs, one per SM, take the units in turn):
//   warp 0      TMA producer: K_j, V_j once per unit; Q_i through an NQ-slot
//               ring and dO_i through an NDO-slot ring (128-byte swizzle)
//   warp 1      allocates 512 TMEM columns; an elected lane issues the five
//               MMAs (the whole warp runs the issue loop)
//   warps 4-11  one thread per query row and half of the key columns (warps
//               4-7: keys 0-63, warps 8-11: keys 64-127): P from S and lse
//               (ex2 with the scale folded in) and dS from dP and D, both
//               written to shared memory as bf16 for the MMAs that read them;
//               between the two, the previous tile's dQ is read out of TMEM,
//               staged (d = 64: in a buffer of its own; d = 128: the first
//               half in the then idle dS buffer, the second after the dS
//               store in the warp's P rows) and added into the fp32
//               dQ accumulator by TMA reduce-add while the tensor core runs
//               the next MMAs
//   warps 2-3   idle
// At the end of a unit warps 4-7 write dV_j and warps 8-11 write scale * dK_j
// (whole rows, through their rows of the P buffer).  Units are dealt to the
// CTAs round-robin in zig-zag (dense, causal) or, with a block mask, handed
// out at run time from a counter (their lengths can differ by dozens of
// times).
// TMEM: S [0,128) dP [128,256) dV [256,256+d) dK [256+d,256+2d);
//       dQ at [384,448) for d = 64 and over the dP columns for d = 128.
#include <math.h>

#include <type_traits>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_philox.cuh"
#include "fa_sched.cuh"

namespace fa {
namespace {

template <int D>
struct BwdSmem {
  static constexpr int CH = D / 64;
  static constexpr int CHUNK = kTile * 128;
  static constexpr int TILE = CH * CHUNK;
  static constexpr int NQ = 2;                  // Q ring (a third slot measured slower)
  static constexpr int NDO = (D == 64) ? 2 : 1;  // dO ring
  static constexpr int PT = 2 * CHUNK;  // 128 x 128 bf16
  static constexpr int K = 0;
  static constexpr int V = K + TILE;
  static constexpr int QR = V + TILE;
  static constexpr int DOR = QR + NQ * TILE;
  static constexpr int P = DOR + NDO * TILE;
  static constexpr int DS = P + PT;
  // d = 64 leaves room for a dQ staging buffer of its own (128 x 64 fp32), so
  // that the wait for the TMA to read it falls a whole step after the reduce
  // is issued; d = 128 stages in the dS buffer
  static constexpr bool OWN_STG = (D == 64);
  static constexpr int STG = DS + PT;
  static constexpr int BAR = STG + (OWN_STG ? 2 * CHUNK : 0);
  static constexpr int B_KV = 0, B_QF = 1, B_QE = B_QF + NQ, B_DOF = B_QE + NQ,
                       B_DOE = B_DOF + NDO, B_SF = B_DOE + NDO, B_DPF = B_SF + 1,
                       B_PR = B_DPF + 1, B_DSR = B_PR + 1, B_DQF = B_DSR + 1, B_DQE = B_DQF + 1,
                       B_FIN = B_DQE + 1, B_SPL = B_FIN + 1, B_EPI = B_SPL + 1;
  // ring of unit indices handed out by the producer (block-sparse kernel)
  static constexpr int NU = 4;
  static constexpr int B_UF = B_EPI + 1, B_UE = B_UF + NU, NBAR = B_UE + NU;
  static constexpr int MISC = BAR + NBAR * 8;
  static constexpr int RING = MISC + 16;  // NU ints
  static constexpr int ALLOC = RING + 4 * NU + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr int T_DQ = (D == 64) ? 384 : T_DP;
};

constexpr int kBwdThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

// A unit's query-tile walk, or a stretch of it: at most `left` more steps.
template <class S>
struct BwdPartSchedule {
  S s;
  int left;
  FA_DEV bool next(int& qt, int& g, const TileLists& L) {
    if (left <= 0) return false;
    --left;
    return s.next(qt, g, L);
  }
};

// Geometry of one work unit: one key/value head x one key tile.
struct BwdUnit {
  int kt;       // key tile
  int N;        // sequence length
  int row0;     // first row of the sequence in its slice
  int zkv;      // key/value slice
  int bq0;      // first query slice of the group
  int bh_base;  // b * H when query slices are heads (variable-length batch)
  int nT;       // tiles of the sequence
};

// Unit u -> its geometry.  False when the key tile lies past the end of its
// (variable-length) sequence; every role of the CTA skips such a unit alike.
template <bool GQA, bool SPARSE>
FA_DEV bool bwd_unit(int u, const BwdParams& p, int Hkv, int G, int ntmax, bool varlen,
                     int nlong, BwdUnit& w) {
  int bkv;
  if (SPARSE) {
    // block mask, key tiles of each head ordered longest first: the nlong
    // long ones of every head come first, rank-major (a kept column of every
    // query tile is a unit as long as dozens of others: started late it
    // would end the kernel late), then the rest head by head, so that one
    // head's Q and dO stay in L2 while its units run
    const int BHkv = p.B * Hkv;
    const int n1 = nlong * BHkv;
    int rank;
    if (u < n1) {
      rank = u / BHkv;
      bkv = u - rank * BHkv;
    } else {
      const int v = u - n1, per = ntmax - nlong;
      bkv = v / per;
      rank = nlong + (v - bkv * per);
    }
    const int hm = p.lists.mask_heads == 1 ? 0 : bkv % p.H;
    w.kt = p.lists.unit_order[hm * ntmax + rank];
  } else {
    bwd_cta_coords(u, p.B * Hkv, ntmax, p.causal != 0, bkv, w.kt);
  }
  w.N = p.N;
  w.row0 = 0;
  w.zkv = bkv;
  w.bq0 = GQA ? (bkv / Hkv) * p.H + (bkv % Hkv) * G : bkv;
  w.bh_base = 0;
  if (varlen) {
    // variable-length batch: slices are heads, sequences are row ranges
    // (indices clamped to [0, total], so bad offsets cannot write outside)
    const int b = bkv / Hkv;
    const int a = min(max(p.cu_seqlens[b], 0), p.total);
    const int e = min(max(p.cu_seqlens[b + 1], a), p.total);
    w.row0 = a;
    w.N = min(e - a, p.N);
    w.zkv = bkv % Hkv;
    w.bq0 = w.zkv * G;
    w.bh_base = b * p.H;
  }
  w.nT = (w.N + kTile - 1) / kTile;
  return w.kt * kTile < w.N;
}

// Persistent: each CTA takes one unit of every round of gridDim.x units.  Per
// unit, K_j and V_j of the next unit load while the previous unit's last dQ
// drains and its dV, dK leave TMEM, and the Q / dO rings and every step
// barrier run on across units.
// DQ = false: no dQ product and no reduce-adds (dQ comes from the query-tile
// pass of the deterministic backward).  SPARSE: a block mask's lists (plain
// kind), units in the lists' longest-first order.  DYN: units handed out at
// run time (block masks, whose units can differ in length by dozens of
// times).  Causal batches keep the zig-zag deal: their unit lengths fall
// evenly, and handing them out at run time measured 4 % slower at d = 128
// (B4 H16 N4096 backward 0.737 -> 0.765 ms, the kernel's registers then
// spill) and no faster at d = 64.
template <int D, int KIND, bool DQ = true, bool SPARSE = false, bool DYN = SPARSE>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdq, const BwdParams p) {
  using L = BwdSmem<D>;
  // with dQ reduce-adds, no early grid_dep_launch: the next kernel may be a
  // preprocess that zeroes the accumulator before its own wait
  if (!DQ) grid_dep_launch();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + L::BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool GQA = KIND != kPlain;
  const int ntmax = (p.N + kTile - 1) / kTile;
  // a unit = one key/value head x one key tile; with grouped K/V it walks
  // the query tiles of every query head of its group (G = H / Hkv)
  // (the plain instantiation carries no group arithmetic)
  const int Hkv = GQA ? p.Hkv : p.H;
  const int G = GQA ? p.H / p.Hkv : 1;
  const int nunits = p.B * Hkv * ntmax;
  constexpr bool DROP = KIND == kGeneralDropout;
  const bool varlen = KIND >= kGeneral && p.cu_seqlens != nullptr;
  const size_t slice_rows = varlen ? static_cast<size_t>(p.total) : static_cast<size_t>(p.N);
  // k-th unit of this CTA: rounds of gridDim.x units, walked left to right in
  // even rounds and right to left in odd ones.  Units come longest first
  // (causal), so each CTA pairs a long unit with a short one.
  auto unit_of = [&](int k) {
    const int base = k * static_cast<int>(gridDim.x);
    return base + ((k & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                           : static_cast<int>(blockIdx.x));
  };
  // block mask: the most long key tiles any mask head has (the same for
  // every role of every CTA), read once the lists are visible (below)
  int nlong = 0;
  auto unit_at = [&](int u, BwdUnit& w) {
    return bwd_unit<GQA, SPARSE>(u, p, Hkv, G, ntmax, varlen, nlong, w);
  };
  // Split last round: when the last round's units fill at most half the
  // grid, each runs as two halves of its query-tile walk on two CTAs.  Only
  // for units of at least 8 steps (the last round's: G x nT dense, G x 1
  // causal, whose last units are the diagonal key tiles): a shorter half
  // pays the unit boundary and the hand-off for too little work (measured:
  // B8 H16 N512 d64, 4-step units, 54 -> 60 us).  Compiled for d = 128
  // only: in the d = 64 kernel the mere run-time option cost the B8 H16
  // N512 backward 52 -> 57 us, though it never split there.
  const int nround = (nunits + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  const int last0 = (nround - 1) * static_cast<int>(gridDim.x);  // first unit of the last round
  const int mlast = nunits - last0;
  const bool split = D == 128 && !DYN && p.part != nullptr && !varlen && nround > 1 &&
                     2 * mlast <= static_cast<int>(gridDim.x) && mlast <= p.nslot &&
                     G * (p.causal ? 1 : ntmax) >= 8;
  // Block mask: units are handed out at run time.  A CTA's first unit is
  // its index; after that the producer takes the next unit index from a
  // counter in the workspace and passes it to the other roles through a
  // ring of NU slots (a slot is refilled once the issuer and all 256
  // compute threads have read it).  Units come in the lists' order (long
  // key tiles first), so the CTAs that draw a long unit take fewer others:
  // with a fixed round-robin deal, a unit as long as dozens of others kept
  // its CTA busy long after the rest had finished.
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::RING);
  const WaitCtl wcu{abort_flag, p.err, p.wait_ns};
  auto dyn_item = [&](int k, int& u) -> bool {
    const int slot = k % L::NU;
    const uint32_t ph = static_cast<uint32_t>(k / L::NU) & 1;
    if (warp == 0) {  // the producer's lane: publish
      if (k >= L::NU && !wait_bar(bar(L::B_UE + slot), ph ^ 1, wcu)) return false;
      int uu = k == 0 ? static_cast<int>(blockIdx.x)
                      : static_cast<int>(gridDim.x) + atomicAdd(p.unit_counter, 1);
      if (uu >= nunits) uu = -1;
      ring[slot] = uu;
      mbar_arrive(bar(L::B_UF + slot));
      u = uu;
      return uu >= 0;
    }
    if (warp == 1) {  // the issuer warp: every lane reads the slot, one arrives
      if (!__all_sync(0xffffffffu, wait_bar(bar(L::B_UF + slot), ph, wcu))) return false;
      u = __shfl_sync(0xffffffffu, ring[slot], 0);
      if (lane == 0) mbar_arrive(bar(L::B_UE + slot));
      return u >= 0;
    }
    if (!wait_bar(bar(L::B_UF + slot), ph, wcu)) return false;
    u = ring[slot];
    mbar_arrive(bar(L::B_UE + slot));
    return u >= 0;
  };
  // k-th item of this CTA: unit u and half uh (-1: the whole unit); false
  // when the CTA has no k-th item
  auto item_of = [&](int k, int& u, int& uh) {
    uh = -1;
    if (DYN) return dyn_item(k, u);
    if (!split || k < nround - 1) {
      u = unit_of(k);
      return u < nunits;
    }
    if (k > nround - 1) return false;
    const int pos = (k & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x)
                            : static_cast<int>(blockIdx.x);
    if (pos >= 2 * mlast) return false;
    u = last0 + pos / 2;
    uh = pos & 1;
    return true;
  };
  // the query-tile walk of item (unit w, half uh): half 0 takes the first
  // half of the unit's steps, half 1 the rest (no block mask here, so a
  // unit has G x (nT, or nT - kt when causal) steps)
  using Sched0 = typename std::conditional<GQA, BwdGroupSchedule, BwdSingleSchedule>::type;
  auto start = [&](const BwdUnit& w, int uh, BwdPartSchedule<Sched0>& ps) {
    ps.s.init(w.kt, w.nT, p.causal != 0, p.lists, w.bq0 % p.H, G);
    ps.left = INT_MAX;
    if (uh >= 0) {
      const int ns = G * (p.causal ? w.nT - w.kt : w.nT);
      int qt, gg;
      if (uh == 1)
        for (int i = 0; i < ns / 2; ++i) ps.s.next(qt, gg, p.lists);
      ps.left = uh ? ns - ns / 2 : ns / 2;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_KV), 1);
    for (int s = 0; s < L::NQ; ++s) {
      mbar_init(bar(L::B_QF + s), 1);
      mbar_init(bar(L::B_QE + s), 1);
    }
    for (int s = 0; s < L::NDO; ++s) {
      mbar_init(bar(L::B_DOF + s), 1);
      mbar_init(bar(L::B_DOE + s), 1);
    }
    mbar_init(bar(L::B_SF), 1);
    mbar_init(bar(L::B_DPF), 1);
    mbar_init(bar(L::B_PR), 256);
    mbar_init(bar(L::B_DSR), 256);
    mbar_init(bar(L::B_DQF), 1);
    mbar_init(bar(L::B_DQE), 256);
    mbar_init(bar(L::B_FIN), 1);
    mbar_init(bar(L::B_SPL), 256);
    mbar_init(bar(L::B_EPI), 256);
    for (int s = 0; s < L::NU; ++s) {
      mbar_init(bar(L::B_UF + s), 1);
      mbar_init(bar(L::B_UE + s), 1 + 256);  // the issuer's lane, the compute threads
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();  // the previous kernel's writes are visible from here on
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.err, p.wait_ns};
  if (SPARSE)
    for (int h = 0; h < p.lists.mask_heads; ++h) nlong = max(nlong, p.lists.nlong[h]);

  using Sched = BwdPartSchedule<Sched0>;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      prefetch_tmap(&tdq);
      uint32_t nq = 0, nd = 0, nkv = 0;  // Q / dO / K-V copies issued
      bool ok = true;
      BwdUnit un;
      // K_j, V_j of the current unit once every product of the previous unit
      // is done (that unit's final commit also follows its own K/V arrival)
      auto load_kv = [&]() -> bool {
        if (nkv > 0 && !wait_bar(bar(L::B_FIN), (nkv - 1) & 1, wc)) return false;
        mbar_arrive_expect_tx(bar(L::B_KV), 2 * L::TILE);
#pragma unroll
        for (int c = 0; c < L::CH; ++c) {
          tma_load_3d(sb + L::K + c * L::CHUNK, &tk, bar(L::B_KV), 64 * c,
                      un.row0 + un.kt * kTile, un.zkv);
          tma_load_3d(sb + L::V + c * L::CHUNK, &tv, bar(L::B_KV), 64 * c,
                      un.row0 + un.kt * kTile, un.zkv);
        }
        ++nkv;
        return true;
      };
      for (int k = 0, u, uh; ok && item_of(k, u, uh); ++k) {
        if (!unit_at(u, un)) continue;
        Sched sch;
        start(un, uh, sch);
        bool kv = false;  // the unit's first Q / dO copies go out before its K/V
        int qt, g;
        while (ok && sch.next(qt, g, p.lists)) {
          const int qpos = nq % L::NQ, dpos = nd % L::NDO;
          const uint32_t qround = nq / L::NQ, dround = nd / L::NDO;
          if (qround > 0 && !wait_bar(bar(L::B_QE + qpos), (qround - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(L::B_QF + qpos), L::TILE);
#pragma unroll
          for (int c = 0; c < L::CH; ++c)
            tma_load_3d(sb + L::QR + qpos * L::TILE + c * L::CHUNK, &tq, bar(L::B_QF + qpos), 64 * c,
                        un.row0 + qt * kTile, un.bq0 + g);
          ++nq;
          if (dround > 0 && !wait_bar(bar(L::B_DOE + dpos), (dround - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(L::B_DOF + dpos), L::TILE);
#pragma unroll
          for (int c = 0; c < L::CH; ++c)
            tma_load_3d(sb + L::DOR + dpos * L::TILE + c * L::CHUNK, &tdo, bar(L::B_DOF + dpos),
                        64 * c, un.row0 + qt * kTile, un.bq0 + g);
          ++nd;
          if (!kv) {
            kv = true;
            if (!(ok = load_kv())) break;
          }
        }
        if (ok && !kv) ok = load_kv();
      }
      // let copies still in flight land before the CTA can exit
      if (nkv > 0) drain_bar(bar(L::B_KV), (nkv - 1) & 1, p.wait_ns);
      if (!ok) {
        const uint32_t fq = nq > static_cast<uint32_t>(L::NQ) ? nq - L::NQ : 0;
        for (uint32_t j = fq; j < nq; ++j)
          drain_bar(bar(L::B_QF + j % L::NQ), (j / L::NQ) & 1, p.wait_ns);
        const uint32_t fd = nd > static_cast<uint32_t>(L::NDO) ? nd - L::NDO : 0;
        for (uint32_t j = fd; j < nd; ++j)
          drain_bar(bar(L::B_DOF + j % L::NDO), (j / L::NDO) & 1, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the issuer: waits and tests are warp votes, so
    // its control flow and operand descriptors are warp-uniform, and the
    // elected lane issues each MMA and commit (a single-lane issuer spent
    // ~90 cycles per MMA instruction).
    {
      auto uwait = [&](uint32_t b, uint32_t ph) {
        return __all_sync(0xffffffffu, wait_bar(b, ph, wc));
      };
      auto utry = [&](uint32_t b, uint32_t ph) { return __all_sync(0xffffffffu, mbar_try(b, ph)); };
      auto ecommit = [&](uint32_t b) {
        if (elect_one()) mma_commit(b);
      };
      constexpr uint32_t idSS = idesc_bf16(128, 128, false, false);  // S, dP
      constexpr uint32_t idTT = idesc_bf16(128, D, true, true);      // dV, dK
      constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);     // dQ
      // One k-step (K = 16) of each product.  The products go out in the
      // order the compute warps consume their results (dV before the next
      // S, dQ before dK at d = 64); only dK and dQ at d = 128 run
      // interleaved k-step by k-step, since dQ's completion may only be
      // signalled with dK's there.
      // X[128 q x 128 k] = A[128 x D] B[128 x D]^T, both K-major
      // operand descriptors: K-major (qk) or MN-major (tt, dq B), advanced per
      // k-step from the descriptor of the operand's first byte
      const uint64_t dk0 = desc_sw128(sb, 16, 1024), dm0 = desc_sw128(sb, L::CHUNK, 1024);
      auto kmaj = [&](uint32_t a) { return desc_advance(dk0, a - sb); };
      auto mnmaj = [&](uint32_t a) { return desc_advance(dm0, a - sb); };
      auto qk_step = [&](uint32_t dst, uint32_t a, uint32_t b, int kk) {
        const uint32_t off = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
        const uint64_t da = kmaj(a + off), db = kmaj(b + off);
        if (elect_one()) mma_bf16_ss(dst, da, db, idSS, kk > 0);
      };
      // Y[128 k x D] += X^T[128 k x 128 q] Z[128 q x D]; X stored [q][k]
      auto tt_step = [&](uint32_t dst, uint32_t x, uint32_t z, bool acc, int kk) {
        const uint64_t da = mnmaj(x + kk * 2048), db = mnmaj(z + kk * 2048);
        if (elect_one()) mma_bf16_ss(dst, da, db, idTT, (acc || kk > 0) ? 1u : 0u);
      };
      // dQ[128 q x D] = dS[128 q x 128 k] K[128 k x D]
      auto dq_step = [&](uint32_t dst, int kk) {
        const uint32_t aoff = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
        const uint64_t da = kmaj(sb + L::DS + aoff), db = mnmaj(sb + L::K + kk * 2048);
        if (elect_one()) mma_bf16_ss(dst, da, db, idDQ, kk > 0);
      };
      auto issue_qk = [&](uint32_t dst, uint32_t a, uint32_t b) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) qk_step(dst, a, b, kk);
      };
      auto issue_tt = [&](uint32_t dst, uint32_t x, uint32_t z, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) tt_step(dst, x, z, acc, kk);
      };
      auto issue_dq = [&](uint32_t dst) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) dq_step(dst, kk);
      };
      const uint32_t tS = tmem + L::T_S, tDP = tmem + L::T_DP, tDV = tmem + L::T_DV,
                     tDK = tmem + L::T_DK, tDQ = tmem + L::T_DQ;
      uint32_t n = 0, ku = 0;  // steps and units so far
      bool ok = true;
      for (int k = 0, u, uh; ok && item_of(k, u, uh); ++k) {
        BwdUnit un;
        if (!unit_at(u, un)) continue;
        Sched sch;
        start(un, uh, sch);
        int qt, qt_n, g_unused;
        ok = uwait(bar(L::B_KV), ku & 1);
        bool have = ok && sch.next(qt, g_unused, p.lists);
        uint32_t nu = 0;  // steps of this unit
        if (ok && have) {
          ok = uwait(bar(L::B_QF + n % L::NQ), (n / L::NQ) & 1);
          if (ok) {
            tc_fence_after();
            issue_qk(tS, sb + L::QR + (n % L::NQ) * L::TILE, sb + L::K);
            ecommit(bar(L::B_SF));
            // d = 128: the previous unit's last dQ shares the dP columns
            if (DQ && D != 64 && n > 0) ok = uwait(bar(L::B_DQE), (n - 1) & 1);
          }
          if (ok) ok = uwait(bar(L::B_DOF + n % L::NDO), (n / L::NDO) & 1);
          if (ok) {
            tc_fence_after();
            issue_qk(tDP, sb + L::DOR + (n % L::NDO) * L::TILE, sb + L::V);
            ecommit(bar(L::B_DPF));
          }
        }
        while (ok && have) {
          const bool have_n = sch.next(qt_n, g_unused, p.lists);
          const uint32_t qpos = n % L::NQ, dpos = n % L::NDO;
          const uint32_t n1 = n + 1;
          // dV += P^T dO_i once P is in shared memory, then the next S when
          // its Q tile is already in (the S columns were read).  dV goes
          // first, not interleaved: its completion releases the P rows that
          // take the pending half of dQ, which the compute warps wait for
          // right after dS (measured 1-1.5 % faster than interleaving)
          if (!(ok = uwait(bar(L::B_PR), n & 1))) break;
          tc_fence_after();
          const uint32_t qn = sb + L::QR + (n1 % L::NQ) * L::TILE;
          const uint32_t dov = sb + L::DOR + dpos * L::TILE;
          issue_tt(tDV, sb + L::P, dov, nu > 0);
          ecommit(bar(L::B_DOE + dpos));
          if (have_n) {
            if (!(ok = uwait(bar(L::B_QF + n1 % L::NQ), (n1 / L::NQ) & 1))) break;
            tc_fence_after();
            issue_qk(tS, qn, sb + L::K);
            ecommit(bar(L::B_SF));
          }
          // dK += dS^T Q_i and dQ_i = dS K once dS is in shared memory.
          // d = 64: dQ first, committed on its own, so that its drain (into a
          // staging buffer of its own) overlaps dK.  d = 128: interleaved,
          // and dQ's completion is signalled only with dK's, because the
          // drain stages dQ in the dS rows that dK reads.
          if (!(ok = uwait(bar(L::B_DSR), n & 1))) break;
          tc_fence_after();
          const uint32_t qv = sb + L::QR + qpos * L::TILE;
          if (!DQ) {
            issue_tt(tDK, sb + L::DS, qv, nu > 0);
            ecommit(bar(L::B_QE + qpos));
          } else if (L::OWN_STG && (n == 0 || utry(bar(L::B_DQE), (n - 1) & 1))) {
            tc_fence_after();
            issue_dq(tDQ);
            ecommit(bar(L::B_DQF));
            issue_tt(tDK, sb + L::DS, qv, nu > 0);
            ecommit(bar(L::B_QE + qpos));
          } else if (!L::OWN_STG) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              tt_step(tDK, sb + L::DS, qv, nu > 0, kk);
              dq_step(tDQ, kk);
            }
            ecommit(bar(L::B_QE + qpos));
            ecommit(bar(L::B_DQF));
          } else {
            issue_tt(tDK, sb + L::DS, qv, nu > 0);
            ecommit(bar(L::B_QE + qpos));
            if (!(ok = uwait(bar(L::B_DQE), (n - 1) & 1))) break;
            tc_fence_after();
            issue_dq(tDQ);
            ecommit(bar(L::B_DQF));
          }
          if (have_n) {
            if (DQ && D != 64) {  // dQ_i shares the dP columns: wait until it is read out
              if (!(ok = uwait(bar(L::B_DQE), n & 1))) break;
              tc_fence_after();
            }
            if (!(ok = uwait(bar(L::B_DOF + n1 % L::NDO), (n1 / L::NDO) & 1))) break;
            tc_fence_after();
            issue_qk(tDP, sb + L::DOR + (n1 % L::NDO) * L::TILE, sb + L::V);
            ecommit(bar(L::B_DPF));
          }
          qt = qt_n;
          have = have_n;
          n = n1;
          ++nu;
        }
        // every product of the unit issued: dV_j, dK_j complete and K_j, V_j
        // free once this lands (also committed on a failed wait, so that the
        // phase count stays that of the other roles).  A unit with no step
        // issued nothing the compute warps gate, so its commit could land
        // right after the previous unit's, two phases ahead of a compute warp
        // still to wait for that one: it waits until they have.
        if (nu == 0 && ku > 0 && !uwait(bar(L::B_EPI), (ku - 1) & 1)) ok = false;
        ecommit(bar(L::B_FIN));
        ++ku;
      }
      if (ku > 0) drain_bar(bar(L::B_FIN), (ku - 1) & 1, p.wait_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------ P, dS, dQ warps
    // Warps 4-7 own key columns [0, 64) of the tile and warps 8-11 own
    // [64, 128); each thread owns one query row (its TMEM lane).  Per query
    // tile: P from S and lse into shared memory, then the previous tile's dQ
    // out of TMEM into the fp32 accumulator (its MMA ran meanwhile), then dS
    // from dP and D into shared memory.  P stays in registers as packed bf16
    // for the dS step.
    const int half = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::T_S + 64 * half;
    const uint32_t tDP = tmem + lane_off + L::T_DP + 64 * half;
    const uint32_t tDQ = tmem + lane_off + L::T_DQ + (D / 2) * half;
    const uint32_t pbuf = sb + L::P + half * L::CHUNK;
    const uint32_t dsbuf = sb + L::DS + half * L::CHUNK;
    const float sl2 = p.scale * kLog2e;
    const DropoutRng rng{p.drop.rk, p.drop.offset, p.drop.t * 0x01010101u};
    bool ok = true;
    uint32_t n = 0, ku = 0;  // steps and units so far
    BwdUnit un{};
    int kbase = 0, kcol0 = 0;  // first key of the tile / of this thread's columns
    auto load_stats = [&](const BwdUnit& w, int t, int gg, float& l_, float& d_) {
      const int row = t * kTile + r;
      const size_t idx =
          static_cast<size_t>(w.bq0 + gg) * slice_rows + w.row0 + (row < w.N ? row : 0);
      l_ = p.lse[idx];
      d_ = p.delta[idx];
    };
    // dQ of query tile t (step m): TMEM -> registers, release the columns,
    // then add this thread's D/2 columns into the fp32 accumulator
    // d = 128: the second 32 columns of this thread's dQ row wait in
    // registers (dq1) until the step's dS is out, then leave through the
    // warp's rows of the P buffer once the dV product has read it; the next
    // P store waits for that read, about a step later.
    // (not with dropout: there the P phase is longer and the deferred half
    // measured slower, 1.81 -> 1.96 ms at B4 H16 N4096)
    constexpr bool SPLIT = (D == 128) && DQ && !DROP;
    uint32_t dq1[32];
    int t1 = 0, g1 = 0;
    bool dq1_live = false;
    auto stage_dq1 = [&]() {
      const uint32_t st1 = pbuf + q4 * 4096;
      // the previous half staged here may still be in flight: at a unit's
      // end two stagings follow each other with no P store between them
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(st1 + sw128_offset(lane, u), dq1[4 * u], dq1[4 * u + 1], dq1[4 * u + 2],
                     dq1[4 * u + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tdq, st1, (D / 2) * half + 32, un.row0 + t1 * kTile + 32 * q4,
                          un.bq0 + g1);
        bulk_commit();
      }
      dq1_live = false;
    };
    // the P rows of this warp may be written once the TMA has read them
    auto p_rows_free = [&]() {
      if (SPLIT) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
    };
    auto drain_dq = [&](uint32_t m, int t, int gg) -> bool {
      if (!__all_sync(0xffffffffu, wait_bar(bar(L::B_DQF), m & 1, wc))) return false;
      tc_fence_after();
      // Reduce-add through the TMA engine: the warp stages its 32 rows x 32
      // columns (4 KB, 128-byte swizzle), for d = 64 in its own staging
      // buffer, for d = 128 (the first 32 of its 64 columns) in its own rows
      // of the dS buffer, which no MMA reads between dQ's completion and the
      // next dS, and lane 0 adds the box into the fp32 accumulator (rows past
      // the tensor are clipped; rows past this sequence but inside the tensor
      // receive exact zeros, since their P and dS rows are 0).
      const uint32_t stage =
          (L::OWN_STG ? sb + L::STG + half * L::CHUNK : dsbuf) + q4 * 4096;
      auto stage_box = [&](const uint32_t (&x)[32], int c) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(stage + sw128_offset(lane, u), x[4 * u], x[4 * u + 1], x[4 * u + 2],
                       x[4 * u + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tdq, stage, (D / 2) * half + 32 * c,
                            un.row0 + t * kTile + 32 * q4, un.bq0 + gg);
          bulk_commit();
        }
      };
      if constexpr (!SPLIT && D == 128) {
        // (d = 128 with dropout) one 32-column box in registers at a time:
        // the first leaves before the second is read, which releases the
        // TMEM columns a little later but keeps the drain within the
        // register budget next to P's packed row
        uint32_t dq[32];
        tmem_ld32(tDQ, dq);
        tmem_ld_wait();
        reg_fence(dq);
        stage_box(dq, 0);
        tmem_ld32(tDQ + 32, dq);
        tmem_ld_wait();
        reg_fence(dq);
        tc_fence_before();
        mbar_arrive(bar(L::B_DQE));
        if (lane == 0) bulk_wait_read_all();  // the first box has been read
        __syncwarp();
        stage_box(dq, 1);
      } else {
        // SPLIT: the second 32 columns go straight into dq1
        constexpr int NCH = SPLIT ? 1 : D / 64;
        uint32_t dq[NCH][32];
#pragma unroll
        for (int c = 0; c < NCH; ++c) tmem_ld32(tDQ + 32 * c, dq[c]);
        if (SPLIT) tmem_ld32(tDQ + 32, dq1);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < NCH; ++c) reg_fence(dq[c]);
        if (SPLIT) reg_fence(dq1);
        tc_fence_before();
        mbar_arrive(bar(L::B_DQE));
        if (SPLIT) {  // second half later, from the P rows
          t1 = t;
          g1 = gg;
          dq1_live = true;
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if (c > 0 || L::OWN_STG) {  // the box staged here before has been read
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          stage_box(dq[c], c);
        }
      }
      // d = 128: the staging rows are this warp's dS rows: the wait for the
      // reads to finish comes just before the next dS store, so that it
      // overlaps the dP wait and the dS arithmetic
      return true;
    };
    // the first of this CTA's items from the k-th on whose unit has keys
    // (k, u, uh updated); false if none
    auto seek = [&](int& k, int& u, int& uh, BwdUnit& w) {
      for (;; ++k) {
        if (!item_of(k, u, uh)) return false;
        if (unit_at(u, w)) return true;
      }
    };
    // current item: its schedule, next query tile and that tile's statistics
    int kc = 0, u = 0, uh = -1;
    bool cur = seek(kc, u, uh, un);
    Sched sch;
    int qt = 0, g = 0;
    bool have = false;
    float lse_c = 0.f, dlt_c = 0.f;
    if (cur) {
      start(un, uh, sch);
      have = sch.next(qt, g, p.lists);
      if (have) load_stats(un, qt, g, lse_c, dlt_c);
    }
    while (ok && cur) {
      kbase = un.kt * kTile;
      kcol0 = kbase + 64 * half;
      const int N = un.N;
      uint32_t nu = 0;  // steps of this unit
      int qt_prev = 0, g_prev = 0;
      while (ok && have) {
        int qt_n = 0, g_n = 0;
        const bool have_n = sch.next(qt_n, g_n, p.lists);
        float lse_n = 0.f, dlt_n = 0.f;
        if (have_n) load_stats(un, qt_n, g_n, lse_n, dlt_n);  // prefetch the next tile's statistics
        const int qrow = qt * kTile + r;
        const bool live = qrow < N && lse_c != -INFINITY;
        const float lse2 = live ? lse_c * kLog2e : 0.f;
        // P = exp2(S * scale * log2e - lse * log2e); masked entries 0
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_SF), n & 1, wc));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[2][32];
        tmem_ld32(tS, sv[0]);
        tmem_ld32(tS + 32, sv[1]);
        tmem_ld_wait();
        reg_fence(sv[0]);
        reg_fence(sv[1]);
        const bool need_mask = (kcol0 + 64 > N) || (p.causal && kcol0 + 63 > qt * kTile);
        // keys kcol0 + i with i >= lim are masked (past N, or after this row
        // when causal)
        int lim = N - kcol0;
        if (p.causal && qrow - kcol0 + 1 < lim) lim = qrow - kcol0 + 1;
        uint32_t pw[32];  // pw[i]: keys 2i, 2i+1 of this thread's 64 columns
        // a row with no live statistics gets the bias -inf: all its P are 0
        const float nb = live ? -lse2 : -INFINITY;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nlse2x2 = f2_pack(nb, nb);
        // scale * S * log2 e - lse * log2 e for two keys in one fp32 x2 FMA
        auto arg2 = [&](int i) {
          return f2_fma(f2_pack(__uint_as_float(sv[i >> 4][(2 * i) & 31]),
                                __uint_as_float(sv[i >> 4][(2 * i + 1) & 31])),
                        sl2x2, nlse2x2);
        };
        if (need_mask) {  // (warp-uniform) the tile crosses N or the diagonal
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float a, b;
            f2_unpack(arg2(i), a, b);
            a = 2 * i < lim ? ex2(a) : 0.f;
            b = 2 * i + 1 < lim ? ex2(b) : 0.f;
            pw[i] = pack_bf16(a, b);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float a, b;
            f2_unpack(arg2(i), a, b);
            pw[i] = pack_bf16(ex2(a), ex2(b));
          }
        }
        // keep bits of this thread's 64 keys (bit k of kb[c]: key 32 c + k)
        uint32_t kb[2] = {0u, 0u};
        p_rows_free();
        if (DROP) {
          // the dV product takes the dropped weights z * P; dS needs P and z
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            const PhiloxOut rw = rng.group((kcol0 >> 4) + g4, qrow, un.bh_base + un.bq0 + g);
            uint32_t mk[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) mk[w] = DropoutRng::keep_bytes(rw.w[w], rng.t4);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t* pp = &pw[8 * g4 + 4 * hh];
              st_shared_v4(pbuf + sw128_offset(r, 2 * g4 + hh), pp[0] & pair_mask(mk[2 * hh], 0),
                           pp[1] & pair_mask(mk[2 * hh], 1), pp[2] & pair_mask(mk[2 * hh + 1], 0),
                           pp[3] & pair_mask(mk[2 * hh + 1], 1));
            }
            kb[g4 >> 1] |= (keep_nibble(mk[0]) | (keep_nibble(mk[1]) << 4) |
                            (keep_nibble(mk[2]) << 8) | (keep_nibble(mk[3]) << 12))
                           << (16 * (g4 & 1));
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_shared_v4(pbuf + sw128_offset(r, u), pw[4 * u], pw[4 * u + 1], pw[4 * u + 2],
                         pw[4 * u + 3]);
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::B_PR));
        if (DQ && nu > 0 && !drain_dq(n - 1, qt_prev, g_prev)) {
          ok = false;
          break;
        }
        // dS = P o (dP - D_i)
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_DPF), n & 1, wc));
        if (!ok) break;
        tc_fence_after();
        const uint64_t dltx2 = f2_pack(dlt_c, dlt_c);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dp[32];
          tmem_ld32(tDP + 32 * c, dp);
          tmem_ld_wait();
          reg_fence(dp);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t pp = pw[16 * c + 4 * g + j];
              float d0 = __uint_as_float(dp[8 * g + 2 * j]);
              float d1 = __uint_as_float(dp[8 * g + 2 * j + 1]);
              if (DROP) {  // dP = z dP~ / (1 - p')
                d0 = ((kb[c] >> (8 * g + 2 * j)) & 1u) ? d0 * p.drop.scale : 0.f;
                d1 = ((kb[c] >> (8 * g + 2 * j + 1)) & 1u) ? d1 * p.drop.scale : 0.f;
              }
              // P o (dP - D) for the two keys: dP - D in fp32 x2, rounded to
              // bf16 (the dS written is bf16 anyway), times the packed bf16 P
              float x0, x1;
              f2_unpack(f2_sub(f2_pack(d0, d1), dltx2), x0, x1);
              w[j] = mul_bf16x2(pp, pack_bf16(x0, x1));
            }
            if (!L::OWN_STG && c == 0 && g == 0) {  // the previous dQ staging in these rows has been read
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
            st_shared_v4(dsbuf + sw128_offset(r, 4 * c + g), w[0], w[1], w[2], w[3]);
          }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::B_DSR));
        if (SPLIT && dq1_live) {  // dV(n) has read P(n): its rows take dQ(n-1)'s second half
          if (!__all_sync(0xffffffffu,
                          wait_bar(bar(L::B_DOE + n % L::NDO), (n / L::NDO) & 1, wc))) {
            ok = false;
            break;
          }
          stage_dq1();
        }
        qt_prev = qt;
        g_prev = g;
        qt = qt_n;
        g = g_n;
        have = have_n;
        lse_c = lse_n;
        dlt_c = dlt_n;
        ++n;
        ++nu;
      }
      if (DQ && ok && nu > 0) ok = drain_dq(n - 1, qt_prev, g_prev);
      if (SPLIT && ok && dq1_live) {  // after the unit's last dV (step n - 1)
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_DOE + (n - 1) % L::NDO),
                                              ((n - 1) / L::NDO) & 1, wc));
        if (ok) stage_dq1();
      }
      // the next unit's schedule and first statistics, loaded while the
      // epilogue runs
      BwdUnit un_n{};
      int k_n = kc + 1, u_n = 0, uh_n = -1;
      const bool cur_n = seek(k_n, u_n, uh_n, un_n);
      Sched sch_n;
      int qt_u = 0, g_u = 0;
      bool have_u = false;
      float lse_u = 0.f, dlt_u = 0.f;
      if (cur_n) {
        start(un_n, uh_n, sch_n);
        have_u = sch_n.next(qt_u, g_u, p.lists);
        if (have_u) load_stats(un_n, qt_u, g_u, lse_u, dlt_u);
      }
      // ---------------------------------------------------- epilogue: dV, dK
      // warps 4-7 write dV_j, warps 8-11 write scale * dK_j; the next unit's
      // first dV, dK products (issued after this thread's next P / dS
      // arrivals) overwrite the columns read here
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_FIN), ku & 1, wc));
      mbar_arrive(bar(L::B_EPI));  // this unit's commit has been seen
      tc_fence_after();
      if (ok) {  // warp-uniform: every lane takes part in the TMEM reads
        const bool dv_side = half == 0;
        const uint32_t tcol = dv_side ? L::T_DV : L::T_DK;
        const float mul = dv_side ? (DROP ? p.drop.scale : 1.f) : p.scale;
        const int krow0 = kbase + 32 * q4;  // key of this warp's first row
        const int nrows = min(32, N - krow0);
        uint8_t* dst = static_cast<uint8_t*>(dv_side ? p.dv : p.dk) +
                       (static_cast<size_t>(un.zkv) * slice_rows + un.row0 + krow0) *
                           static_cast<size_t>(D) * 2;
        // Each thread packs 64 columns of its key row (128 bytes) into this
        // warp's 32 rows of the P buffer (the unit's last dV product, which
        // read it, has completed); then each store writes 4 whole rows.
        const uint32_t stg = pbuf + q4 * 4096;
        p_rows_free();
        // Half of a split unit: the first half to finish (order 0) parks its
        // fp32 rows in the unit's slot and raises the slot's ready flag; the
        // second (order 1) adds them to its own and writes the unit's rows.
        int order = -1;
        float* prow = nullptr;  // this thread's row in the slot
        int* ready = nullptr;
        if (uh >= 0) {
          const int slot = u - last0;
          ready = p.part_cnt + p.nslot + slot;
          prow = p.part + (static_cast<size_t>(slot) * 2 + (dv_side ? 0 : 1)) * kTile * D +
                 static_cast<size_t>(r) * D;
          volatile int* sorder = reinterpret_cast<volatile int*>(smem + L::MISC + 8);
          if (threadIdx.x == 128) *sorder = atomicAdd(p.part_cnt + slot, 1);
          mbar_arrive(bar(L::B_SPL));  // phase 0: the order is published
          ok = __all_sync(0xffffffffu, wait_bar(bar(L::B_SPL), 0, wc));
          order = *sorder;
          if (ok && order == 1) {  // the other half's rows are in the slot
            bool seen = false;
            const uint64_t t0 = global_ns();
            while (!(seen = ld_acquire_gpu(ready) != 0) && !*wc.abort &&
                   global_ns() - t0 <= wc.limit_ns) {
            }
            if (!seen) {
              *wc.abort = 1;
              atomicCAS(wc.err, kDevOk, kDevTimeout);
            }
            ok = __all_sync(0xffffffffu, seen);
          }
        }
#pragma unroll 1
        for (int c = 0; ok && c < D / 64; ++c) {
          uint32_t a[2][32];
          if (nu > 0) {
            tmem_ld32(tmem + lane_off + tcol + 64 * c, a[0]);
            tmem_ld32(tmem + lane_off + tcol + 64 * c + 32, a[1]);
            tmem_ld_wait();
            reg_fence(a[0]);
            reg_fence(a[1]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) a[0][j] = a[1][j] = 0u;
          }
          if (order == 0) {  // park 64 columns of this row, no output
            float4* pr = reinterpret_cast<float4*>(prow + 64 * c);
#pragma unroll
            for (int v = 0; v < 16; ++v)
              pr[v] = make_float4(__uint_as_float(a[v >> 3][4 * (v & 7)]),
                                  __uint_as_float(a[v >> 3][4 * (v & 7) + 1]),
                                  __uint_as_float(a[v >> 3][4 * (v & 7) + 2]),
                                  __uint_as_float(a[v >> 3][4 * (v & 7) + 3]));
            continue;
          }
          if (order == 1) {  // add the parked half
            const float4* pr = reinterpret_cast<const float4*>(prow + 64 * c);
#pragma unroll
            for (int v = 0; v < 16; ++v) {
              const float4 o = __ldcg(pr + v);
              uint32_t* x = &a[v >> 3][4 * (v & 7)];
              x[0] = __float_as_uint(__uint_as_float(x[0]) + o.x);
              x[1] = __float_as_uint(__uint_as_float(x[1]) + o.y);
              x[2] = __float_as_uint(__uint_as_float(x[2]) + o.z);
              x[3] = __float_as_uint(__uint_as_float(x[3]) + o.w);
            }
          }
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint32_t* x = &a[v >> 2][8 * (v & 3)];
            st_shared_v4(stg + sw128_offset(lane, v),
                         pack_bf16(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul),
                         pack_bf16(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul),
                         pack_bf16(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul),
                         pack_bf16(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul));
          }
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int j = 4 * it + (lane >> 3), cc = lane & 7;
            const uint4 v = ld_shared_v4(stg + sw128_offset(j, cc));
            if (j < nrows)
              *reinterpret_cast<uint4*>(dst + static_cast<size_t>(j) * D * 2 + c * 128 + cc * 16) = v;
          }
          __syncwarp();
        }
        if (ok && order == 0) {  // phase 1: every row parked, then the flag
          mbar_arrive(bar(L::B_SPL));
          if (threadIdx.x == 128) {
            if (wait_bar(bar(L::B_SPL), 1, wc)) {
              __threadfence();
              st_release_gpu(ready, 1);
            }
          }
        }
      }
      tc_fence_before();
      ++ku;
      kc = k_n;
      u = u_n;
      uh = uh_n;
      cur = cur_n;
      un = un_n;
      sch = sch_n;
      qt = qt_u;
      g = g_u;
      have = have_u;
      lse_c = lse_u;
      dlt_c = dlt_u;
    }
    if (lane == 0) bulk_wait_all();  // every dQ reduce of this warp has landed
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int KIND, bool DQ = true, bool SPARSE = false, bool DYN = SPARSE>
cudaError_t launch_bwd_d(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                         cudaStream_t stream) {
  using L = BwdSmem<D>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(
      attr_done, reinterpret_cast<const void*>(fa_bwd_kernel<D, KIND, DQ, SPARSE, DYN>),
      L::ALLOC);
  if (e != cudaSuccess) return e;
  const int nT = (p.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(nT) * p.B * (p.Hkv > 0 ? p.Hkv : p.H);
  // persistent: one CTA per SM (the CTA holds the SM's TMEM and most of its
  // shared memory), each walking units blockIdx.x, blockIdx.x + grid, ...
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const long long ctas = units < sms ? units : sms;
  return launch_pdl(fa_bwd_kernel<D, KIND, DQ, SPARSE, DYN>, dim3(static_cast<unsigned>(ctas)),
                    dim3(kBwdThreads), L::ALLOC, stream, tq, tk, tv, tdo, tdq, p);
}

}  // namespace

cudaError_t launch_backward_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo,
                                 const CUtensorMap& tdq, cudaStream_t stream) {
  const int kind = p.drop.t ? kGeneralDropout
                   : p.cu_seqlens ? kGeneral
                   : (p.Hkv > 0 && p.Hkv != p.H) ? kGrouped : kPlain;
  if (p.skip_dq) {  // deterministic backward: plain layout only
    if (kind != kPlain) return cudaErrorInvalidValue;
    if (p.d == 64) return launch_bwd_d<64, kPlain, false>(p, tq, tk, tv, tdo, tdq, stream);
    if (p.d == 128) return launch_bwd_d<128, kPlain, false>(p, tq, tk, tv, tdo, tdq, stream);
    return cudaErrorInvalidValue;
  }
  if (p.lists.col_ptr != nullptr) {  // block mask: plain layout only
    if (kind != kPlain || p.lists.unit_order == nullptr || p.lists.nlong == nullptr)
      return cudaErrorInvalidValue;
    if (p.d == 64) return launch_bwd_d<64, kPlain, true, true>(p, tq, tk, tv, tdo, tdq, stream);
    if (p.d == 128) return launch_bwd_d<128, kPlain, true, true>(p, tq, tk, tv, tdo, tdq, stream);
    return cudaErrorInvalidValue;
  }
  if (p.d == 64) {
    if (kind == kGeneralDropout)
      return launch_bwd_d<64, kGeneralDropout>(p, tq, tk, tv, tdo, tdq, stream);
    if (kind == kGeneral) return launch_bwd_d<64, kGeneral>(p, tq, tk, tv, tdo, tdq, stream);
    if (kind == kGrouped) return launch_bwd_d<64, kGrouped>(p, tq, tk, tv, tdo, tdq, stream);
    return launch_bwd_d<64, kPlain>(p, tq, tk, tv, tdo, tdq, stream);
  }
  if (p.d == 128) {
    if (kind == kGeneralDropout)
      return launch_bwd_d<128, kGeneralDropout>(p, tq, tk, tv, tdo, tdq, stream);
    if (kind == kGeneral) return launch_bwd_d<128, kGeneral>(p, tq, tk, tv, tdo, tdq, stream);
    if (kind == kGrouped) return launch_bwd_d<128, kGrouped>(p, tq, tk, tv, tdo, tdq, stream);
    return launch_bwd_d<128, kPlain>(p, tq, tk, tv, tdo, tdq, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
