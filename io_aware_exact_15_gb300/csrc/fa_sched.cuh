// Tile schedules: which key tiles a forward CTA visits and which query tiles
// a backward CTA visits.  Every role of a CTA (TMA producer, MMA issuer,
// softmax warps) walks its own copy of the same deterministic sequence.
//
// Forward CTA = one head x a pair of query tiles (qt0 = 2*pair, qt1 = qt0+1);
// the two tiles share each key/value tile they both need.  Each step yields
// a key tile kt and a membership mask (bit s: query tile s uses kt).
//   dense     : kt = 0 .. nT-1
//   causal    : kt = 0 .. qt1 (tile qt0 stops at kt = qt0): k-tile j holds an
//               allowed element of query tile i iff j <= i (Br = Bc), which
//               gives n(n+1)/2 tiles per head for n query tiles
//   sparse    : merge of the two ascending CSR lists of the block mask,
//               intersected with the causal rule when both apply
// Backward CTA = one head x one key tile kt; the query tiles it visits are
// kt .. nT-1 (causal), 0 .. nT-1 (dense) or the ascending CSC list.
#pragma once

#include <limits.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

// BC: keys per key tile.  Query tiles are always kTile = 128 rows; the key
// tile width differs from 128 only in the block-size sweep (dense and causal
// batches): key tile j of width BC holds an allowed key of query tile i iff
// j * BC <= 128 * i + 127.  Block masks (128 x 128 tiles) need BC = 128.
template <int BC>
struct FwdScheduleT {
  int qt[2];
  bool act[2];
  bool causal, sparse;
  const int* la;
  const int* lb;
  int na, nb, ia, ib;
  int next_dense, end_dense;

  // last key tile that query tile t reaches under the causal rule
  static FA_DEV int causal_last(int t) {
    if constexpr (BC == kTile) return t;
    return (kTile * t + kTile - 1) / BC;
  }

  // single: the CTA takes one query tile (index `pair`) instead of two;
  // nT: query tiles of the sequence (key tiles: ceil(nT * 128 / BC))
  FA_DEV void init(int pair, int nT, bool causal_, const TileLists& L, int head,
                   bool single = false, int nkt = -1) {
    qt[0] = single ? pair : 2 * pair;
    qt[1] = qt[0] + 1;
    act[0] = true;
    act[1] = !single && qt[1] < nT;
    causal = causal_;
    sparse = BC == kTile && L.row_ptr != nullptr;
    next_dense = 0;
    end_dense = 0;
    la = lb = nullptr;
    na = nb = ia = ib = 0;
    if (!sparse) {
      if (nkt < 0) nkt = BC == kTile ? nT : (nT * kTile + BC - 1) / BC;
      end_dense = causal ? causal_last(act[1] ? qt[1] : qt[0]) + 1 : nkt;
      if (end_dense > nkt) end_dense = nkt;
      return;
    }
    const int hm = (L.mask_heads == 1) ? 0 : head;
    const int* rp = L.row_ptr + static_cast<size_t>(hm) * (nT + 1);
    const int* ci = L.col_idx + static_cast<size_t>(hm) * nT * nT;
    la = ci + rp[qt[0]];
    na = rp[qt[0] + 1] - rp[qt[0]];
    if (act[1]) {
      lb = ci + rp[qt[1]];
      nb = rp[qt[1] + 1] - rp[qt[1]];
    } else {
      lb = la;
      nb = 0;
    }
    if (causal) {
      while (na > 0 && la[na - 1] > qt[0]) --na;
      while (nb > 0 && lb[nb - 1] > qt[1]) --nb;
    }
  }

  FA_DEV bool next(int& kt, int& mem) {
    if (!sparse) {
      if (next_dense >= end_dense) return false;
      kt = next_dense++;
      mem = ((!causal || kt <= causal_last(qt[0])) ? 1 : 0) |
            ((act[1] && (!causal || kt <= causal_last(qt[1]))) ? 2 : 0);
      return true;
    }
    const int ka = ia < na ? la[ia] : INT_MAX;
    const int kb = ib < nb ? lb[ib] : INT_MAX;
    kt = ka < kb ? ka : kb;
    if (kt == INT_MAX) return false;
    mem = 0;
    if (ka == kt) {
      mem |= 1;
      ++ia;
    }
    if (kb == kt) {
      mem |= 2;
      ++ib;
    }
    return true;
  }
};

using FwdSchedule = FwdScheduleT<kTile>;

struct BwdSchedule {
  bool sparse;
  const int* lst;
  int nl, pos;
  int next_dense, end_dense;

  FA_DEV void init(int kt, int nT, bool causal, const TileLists& L, int head) {
    sparse = L.col_ptr != nullptr;
    lst = nullptr;
    nl = pos = 0;
    next_dense = causal ? kt : 0;
    end_dense = nT;
    if (!sparse) return;
    const int hm = (L.mask_heads == 1) ? 0 : head;
    const int* cp = L.col_ptr + static_cast<size_t>(hm) * (nT + 1);
    lst = L.row_idx + static_cast<size_t>(hm) * nT * nT + cp[kt];
    nl = cp[kt + 1] - cp[kt];
    if (causal)
      while (pos < nl && lst[pos] < kt) ++pos;
  }

  FA_DEV bool next(int& qt) {
    if (!sparse) {
      if (next_dense >= end_dense) return false;
      qt = next_dense++;
      return true;
    }
    if (pos >= nl) return false;
    qt = lst[pos++];
    return true;
  }
};

// Backward schedule of a key/value head shared by G query heads (grouped
// K/V): the query tiles of query head hq0, then those of hq0 + 1, ...  Each
// step yields (query tile, group member g).  G = 1 is the plain schedule.
struct BwdGroupSchedule {
  BwdSchedule s;
  int g, G, kt, nT, hq0;
  bool causal;

  FA_DEV void init(int kt_, int nT_, bool causal_, const TileLists& L, int hq0_, int G_) {
    kt = kt_;
    nT = nT_;
    causal = causal_;
    hq0 = hq0_;
    G = G_;
    g = 0;
    s.init(kt, nT, causal, L, hq0);
  }

  // L: the same lists init() was given
  FA_DEV bool next(int& qt, int& gout, const TileLists& L) {
    for (;;) {
      if (s.next(qt)) {
        gout = g;
        return true;
      }
      if (++g >= G) return false;
      s.init(kt, nT, causal, L, hq0 + g);
    }
  }
};

// The plain schedule behind the grouped interface (a group of one).
struct BwdSingleSchedule {
  BwdSchedule s;
  FA_DEV void init(int kt, int nT, bool causal, const TileLists& L, int head, int) {
    s.init(kt, nT, causal, L, head);
  }
  FA_DEV bool next(int& qt, int& g, const TileLists&) {
    g = 0;
    return s.next(qt);
  }
};

// CTA index -> (head, query-tile pair) for the forward grid.  Causal CTAs
// are issued longest-first (largest pair index first, all heads of one rank
// together); dense CTAs go head by head so a head's K/V stay in L2.
FA_DEV void fwd_cta_coords(int cta, int BH, int npairs, bool causal, int& bh, int& pair) {
  if (causal) {
    const int rank = cta / BH;
    bh = cta - rank * BH;
    pair = npairs - 1 - rank;
  } else {
    bh = cta / npairs;
    pair = cta - bh * npairs;
  }
}

// CTA index -> (head, key tile) for the backward grid; causal key tile j has
// nT - j query tiles, so small j (most work) is issued first.
FA_DEV void bwd_cta_coords(int cta, int BH, int nT, bool causal, int& bh, int& kt) {
  if (causal) {
    kt = cta / BH;
    bh = cta - kt * BH;
  } else {
    bh = cta / nT;
    kt = cta - bh * nT;
  }
}

}  // namespace fa
