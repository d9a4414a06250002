// Host-only check of the persistent scans' work plans (the plan helpers of
// the kernels' internal header): for a shape given on the command line it
// walks every CTA range item by item, as the kernels do, and checks that
//   - the items cover every (sequence, chunk) unit exactly once;
//   - an item's piece index and chunk range agree with the piece table
//     (plan_pieces / plan_piece_range), whose pieces tile each sequence in
//     time order;
//   - no range is longer than ceil(U / P) chunks (the balance the plan
//     promises), and every range but possibly empty tail ranges has work;
//   - the aggregate pass's slots (agg_slot) cover the chunks of the later
//     pieces (k >= 1) exactly once, in sub-pieces of at most kAggSub chunks
//     that lie inside one piece, with slots inside [0, agg_slots) that grow
//     with time, and agree with agg_piece_slots.
// Prints "ok <U> <P> <H> <maxp> <agg chunks>" or the first violation (exit 1).
// Usage: plan_check B L D N [sms]
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "s6_internal.cuh"

namespace s6 {
BwdPlan bwd_plan(int B, int L, int D, int N, int sms);
}

static int fail(const char* what, long long a, long long b, long long c) {
  std::printf("FAIL %s (%lld %lld %lld)\n", what, a, b, c);
  return 1;
}

int main(int argc, char** argv) {
  if (argc < 5) return fail("usage", 0, 0, 0);
  const int B = std::atoi(argv[1]), L = std::atoi(argv[2]), D = std::atoi(argv[3]), N = std::atoi(argv[4]);
  const int sms = argc > 5 ? std::atoi(argv[5]) : 152;
  const s6::BwdPlan pl = s6::bwd_plan(B, L, D, N, sms);
  const long long nseq = s6::plan_nseq(pl);
  if (nseq * pl.nch != pl.U) return fail("U != nseq * nch", pl.U, nseq, pl.nch);
  // the piece table: pieces tile each sequence in time order
  for (long long s = 0; s < nseq; ++s) {
    const int K = s6::plan_pieces(pl, s);
    if (K < 1 || K > pl.maxp) return fail("piece count", s, K, pl.maxp);
    int at = 0;
    for (int k = 0; k < K; ++k) {
      int lo, hi;
      s6::plan_piece_range(pl, s, k, lo, hi);
      if (lo != at || hi <= lo) return fail("piece range", s, k, lo);
      at = hi;
    }
    if (at != pl.nch) return fail("pieces end", s, at, pl.nch);
  }
  // walk the ranges
  std::vector<int> seen((size_t)pl.U, 0);
  const long long cap = (pl.U + pl.P - 1) / pl.P;
  for (int w = 0; w < pl.P; ++w) {
    const long long ub = s6::plan_bound(pl, w), ue = s6::plan_bound(pl, w + 1);
    if (ue < ub || ue - ub > cap) return fail("range length", w, ub, ue);
    for (long long u = ub, next; u < ue; u = next) {
      long long sq;
      int c_lo, c_hi, k;
      s6::plan_item(pl, u, ue, sq, c_lo, c_hi, k, next);
      if (next <= u || next > ue || sq < 0 || sq >= nseq) return fail("item", w, u, next);
      if (c_hi - c_lo != next - u) return fail("item length", w, u, c_hi - c_lo);
      int lo, hi;
      s6::plan_piece_range(pl, sq, k, lo, hi);
      if (k < 0 || k >= s6::plan_pieces(pl, sq) || lo != c_lo || hi != c_hi) return fail("item piece", sq, k, c_lo);
      for (int c = c_lo; c < c_hi; ++c) {
        int& v = seen[(size_t)(sq * pl.nch + c)];
        if (v++) return fail("unit twice", sq, c, w);
      }
    }
  }
  for (long long i = 0; i < pl.U; ++i)
    if (seen[(size_t)i] != 1) return fail("unit missed", i / pl.nch, i % pl.nch, 0);
  // the aggregate pass's sub-pieces
  long long agg = 0;
  const int nslot = pl.maxp > 1 ? s6::agg_slots(pl) : 0;
  for (long long s = 0; s < nseq; ++s) {
    std::vector<int> cov((size_t)pl.nch, 0);
    int last_z = -1, last_end = -1;
    for (int z = 0; z < nslot; ++z) {
      int k, cs, ce;
      if (!s6::agg_slot(pl, s, z, k, cs, ce)) continue;
      int lo, hi;
      s6::plan_piece_range(pl, s, k, lo, hi);
      if (k < 1 || cs < lo || ce > hi || ce - cs > s6::kAggSub || ce <= cs) return fail("sub-piece", s, z, cs);
      if (cs < last_end || z <= last_z) return fail("slot order", s, z, cs);
      int z0, z1;
      s6::agg_piece_slots(pl, s, k, z0, z1);
      if (z < z0 || z > z1 || z1 >= nslot) return fail("piece slots", s, z, z1);
      last_z = z;
      last_end = ce;
      for (int c = cs; c < ce; ++c) cov[(size_t)c]++;
      agg += ce - cs;
    }
    const int K = s6::plan_pieces(pl, s);
    for (int k = 0; k < K; ++k) {
      int lo, hi;
      s6::plan_piece_range(pl, s, k, lo, hi);
      for (int c = lo; c < hi; ++c)
        if (cov[(size_t)c] != (k >= 1 ? 1 : 0)) return fail("aggregate cover", s, k, c);
      if (k >= 1) {  // a piece's slots are all used
        int z0, z1;
        s6::agg_piece_slots(pl, s, k, z0, z1);
        for (int z = z0; z <= z1; ++z) {
          int kk, cs, ce;
          if (!s6::agg_slot(pl, s, z, kk, cs, ce) || kk != k) return fail("empty slot", s, k, z);
        }
      }
    }
  }
  std::printf("ok %lld %d %d %d %lld\n", pl.U, pl.P, pl.H, pl.maxp, agg);
  return 0;
}
