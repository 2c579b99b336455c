// Expert-parallel dispatch plan: the host-side contracts of the MoonEP page
// ("Step-by-step") for a layer whose E experts are spread over R ranks.
//
//   * Every rank processes exactly S*K routed rows, S tokens per rank and K
//     experts per token, whatever the router's skew.
//   * Each rank holds its own group of G = E/R experts (rank r: experts
//     [rG, rG + G)) plus a preload pool of B slots for copies of experts of
//     other ranks; with B = E/R any whole remote group fits.
//   * The local weight tensor is one contiguous [G + B, H, H'] block per
//     projection (home experts, then the slots), and the rows a rank receives
//     are addressed by a local cu_seqlens of G + B + 1 entries.
//   * The gradient of a slot is kept apart from the home gradient; reduce_grad
//     reads the slots holding copies of a home expert on every rank, adds them
//     to the home gradient and clears them.
//
// The page fixes these contracts but not the scheduler.  The one here: lay
// all R*S*K routed pairs out in expert order (source rank, then the source's
// pair order, inside an expert) and give rank d the d-th run of S*K of them.
// With balanced routing every rank's run is exactly its home group; skew
// shifts the runs, so a rank takes the boundary experts of the neighbouring
// groups.  A rank's remote experts fill its slots in decreasing order of rows
// (ties: lower expert first); rows of remote experts left without a slot are
// counted as remote reads (the page's fallback: weights read from the home
// rank through symmetric memory, slower but correct).  The plan depends only
// on the counts, so every rank computes the same plan from the gathered
// counts without further communication.
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "moe_internal.cuh"

extern "C" {

int moe_ep_plan(int R, int E, int S, int K, int B, const int32_t* counts, int32_t* piece_count,
                int32_t* piece_offset, int32_t* slot_expert, int32_t* local_counts, int32_t* remote_reads) {
  if (R < 1 || E < 1 || E % R != 0 || S < 0 || K < 1 || K > E || B < 0) return MOE_ERR_INVALID_ARG;
  if (!counts || !piece_count || !piece_offset || !local_counts || !remote_reads || (B > 0 && !slot_expert))
    return MOE_ERR_INVALID_ARG;
  const long long SK = (long long)S * K;
  if (SK > 0x7fffffffLL || (long long)R * R * E > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  const int G = E / R;
  for (int s = 0; s < R; ++s) {
    long long row = 0;
    for (int e = 0; e < E; ++e) {
      const int32_t c = counts[(long long)s * E + e];
      if (c < 0) return MOE_ERR_INVALID_ARG;
      row += c;
    }
    if (row != SK) return MOE_ERR_INVALID_ARG;  // every source rank routes exactly S*K pairs
  }
  // start of bucket (s, e) in the expert-ordered layout of all pairs
  std::vector<long long> start((size_t)R * E);
  long long pos = 0;
  for (int e = 0; e < E; ++e)
    for (int s = 0; s < R; ++s) {
      start[(size_t)s * E + e] = pos;
      pos += counts[(long long)s * E + e];
    }
  std::vector<long long> rows_of((size_t)E);
  std::vector<std::pair<long long, int>> remote;
  for (int d = 0; d < R; ++d) {
    const long long lo_d = d * SK, hi_d = lo_d + SK;
    std::fill(rows_of.begin(), rows_of.end(), 0);
    for (int s = 0; s < R; ++s)
      for (int e = 0; e < E; ++e) {
        const size_t b = (size_t)s * E + e;
        const long long lo = std::max(start[b], lo_d);
        const long long hi = std::min(start[b] + counts[b], hi_d);
        const long long c = hi > lo ? hi - lo : 0;
        const size_t o = ((size_t)d * R + s) * E + e;
        piece_count[o] = (int32_t)c;
        piece_offset[o] = (int32_t)(c ? lo - start[b] : 0);
        rows_of[e] += c;
      }
    int32_t* lc = local_counts + (size_t)d * (G + B);
    for (int i = 0; i < G + B; ++i) lc[i] = 0;
    for (int i = 0; i < G; ++i) lc[i] = (int32_t)rows_of[(size_t)d * G + i];
    remote.clear();
    for (int e = 0; e < E; ++e)
      if (e / G != d && rows_of[e] > 0) remote.emplace_back(-rows_of[e], e);
    std::sort(remote.begin(), remote.end());  // most rows first, then lower expert
    long long rr = 0;
    for (int j = 0; j < B; ++j) slot_expert[(size_t)d * B + j] = -1;
    for (size_t i = 0; i < remote.size(); ++i) {
      if ((int)i < B) {
        slot_expert[(size_t)d * B + i] = remote[i].second;
        lc[G + i] = (int32_t)(-remote[i].first);
      } else {
        rr += -remote[i].first;
      }
    }
    remote_reads[d] = (int32_t)rr;
  }
  return MOE_OK;
}

}  // extern "C"
