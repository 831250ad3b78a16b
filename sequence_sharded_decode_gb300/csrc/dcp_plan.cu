// Work planning on the device: lanes, tiles and the balanced split over CTAs.
//
// One CTA of 1024 threads reads the per-sequence lengths and shard ranges
// (device memory, so the host never synchronises), and writes into the
// workspace:
//   lanes[l]   token range, tile count, and the items covering the lane
//   items[k]   (lane, tile range, output row) in layout order
//   cta_begin  CTA c processes items [cta_begin[c], cta_begin[c+1])
//   groups[r]  (group order only) the CTA runs row group r spans, its
//              workspace rows, and zeroed piece counters
//   finish     (group order only) the row groups the MLA one-call path
//              finishes in a kernel of its own: no tokens, or more than
//              kMlaMergeInKernel pieces
// CTA c's tiles are [c*T/S, (c+1)*T/S) of the T tiles laid end to end, so the
// CTAs' loads differ by at most one tile. With gangs (the many-row GQA kernel:
// `gang` token groups of one KV range), a "CTA" of the plan is a gang of CTAs
// that run the same items, each on its own token group's lane, so the gang
// reads every K/V tile at about the same time and it leaves HBM about once.
#include <climits>

#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr int kPlanThreads = 1024;

struct Scan2 {
  long long a, b;
};

// Block-wide exclusive scan of two int64 values per thread; returns the
// exclusive prefix for this thread and writes the block totals.
__device__ Scan2 block_exclusive_scan2(Scan2 v, Scan2* totals) {
  __shared__ long long sa[32], sb[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long ia = v.a, ib = v.b;
  for (int o = 1; o < 32; o <<= 1) {
    long long ta = __shfl_up_sync(0xffffffffu, ia, o);
    long long tb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += ta; ib += tb; }
  }
  if (lane == 31) { sa[warp] = ia; sb[warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    long long wa = sa[lane], wb = sb[lane];
    for (int o = 1; o < 32; o <<= 1) {
      long long ta = __shfl_up_sync(0xffffffffu, wa, o);
      long long tb = __shfl_up_sync(0xffffffffu, wb, o);
      if (lane >= o) { wa += ta; wb += tb; }
    }
    sa[lane] = wa;
    sb[lane] = wb;
  }
  __syncthreads();
  Scan2 r;
  const long long pa = warp ? sa[warp - 1] : 0, pb = warp ? sb[warp - 1] : 0;
  r.a = pa + ia - v.a;
  r.b = pb + ib - v.b;
  totals->a = sa[31];
  totals->b = sb[31];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void unit_range(const RangeSpec& rs, int u, int* lo, int* hi, int* start) {
  const int i = u / rs.B, r = u - i * rs.B;
  const int G = (rs.qlen + rs.tpr - 1) / rs.tpr;
  const int b = r / G, k = r - b * G;
  const int j_last = min(rs.qlen, (k + 1) * rs.tpr) - 1;  // last query token of the group
  int L = rs.seq_lens[b] - (rs.qlen - 1 - j_last);         // its causal limit
  if (L < 0) L = 0;
  int s, e;
  if (rs.mode == 0) {
    s = rs.starts[b * rs.N + i];
    e = (i + 1 < rs.N) ? rs.starts[b * rs.N + i + 1] : INT_MAX;
  } else {
    s = rs.range[2 * b];
    e = rs.range[2 * b + 1];
  }
  if (s < 0) {  // a shard cannot start before position 0: flag it, attend nothing
    raise_flag(rs.err, DCP_DEVERR_POSITION);
    s = 0;
    e = 0;
  }
  int l = s;
  if (l > L) l = L;
  int h = e < L ? e : L;
  if (h < l) h = l;
  *lo = l;
  *hi = h;
  *start = s;
}

// CTA that owns flattened tile x: the largest c with floor(c*T/S) <= x.
__device__ __forceinline__ int cta_of(long long x, long long T, long long S) {
  return (int)(((x + 1) * S - 1) / T);
}
__device__ __forceinline__ long long cta_start(long long c, long long T, long long S) {
  return c * T / S;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(RangeSpec rs, int lanes_per_unit, int tile,
                                                            int n_ctas, char* ws, WsLayout L, int group_order,
                                                            int gang) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  LaneRec* lanes = reinterpret_cast<LaneRec*>(ws + L.lanes_off);
  ItemRec* items = reinterpret_cast<ItemRec*>(ws + L.items_off);
  int* cta_begin = reinterpret_cast<int*>(ws + L.cta_off);
  GroupRec* groups = reinterpret_cast<GroupRec*>(ws + L.grp_off);
  int* finish = reinterpret_cast<int*>(ws + L.fin_off);
  long long n_finish = 0;

  const int n_lanes = rs.B * rs.N * lanes_per_unit;
  const int group_lanes = rs.N * lanes_per_unit;  // lanes of one row group
  const int G = (rs.qlen + rs.tpr - 1) / rs.tpr;  // token groups per sequence
  const int n_work = n_lanes / gang;              // laid-out work units: lanes, or gangs of lanes
  // the (first) lane of the work unit at layout position x: shard by shard (x
  // itself), row group by row group (x = (r * N + shard) * lanes_per_unit + j),
  // or (gang > 1) gang by gang: the lanes of token groups kb * gang .. kb *
  // gang + gang - 1 of one (shard, sequence, KV head), lanes_per_unit apart
  auto lane_at = [&](int x) {
    if (group_order) {
      const int r = x / group_lanes, rem = x - r * group_lanes;
      const int i = rem / lanes_per_unit, j = rem - i * lanes_per_unit;
      return (i * rs.B + r) * lanes_per_unit + j;
    }
    if (gang == 1) return x;
    const int kvh = x % lanes_per_unit, rest = x / lanes_per_unit;
    const int per_seq = G / gang, sb = rest / per_seq, kb = rest - sb * per_seq;  // sb = shard * seqs + b
    return (sb * G + kb * gang) * lanes_per_unit + kvh;
  };
  const int per = (n_work + kPlanThreads - 1) / kPlanThreads;
  const int x0 = threadIdx.x * per;
  const int x1 = min(n_work, x0 + per);

  // pass 1: ranges and tile counts. A gang's lanes (one KV range, causal
  // limits a token group apart) all take the union of their non-empty ranges:
  // their rows are masked at their own tokens' limits anyway.
  long long my_tiles = 0;
  for (int x = x0; x < x1; ++x) {
    const int l0 = lane_at(x);
    int lo_u = 0, hi_u = 0, start_u = 0;
    bool any = false;
    for (int m = 0; m < gang; ++m) {
      int lo, hi, start;
      unit_range(rs, (l0 + m * lanes_per_unit) / lanes_per_unit, &lo, &hi, &start);
      if (hi > lo) {
        lo_u = any ? min(lo_u, lo) : lo;
        hi_u = any ? max(hi_u, hi) : hi;
        start_u = start;
        any = true;
      } else if (m == 0) {
        lo_u = lo;
        hi_u = hi;
        start_u = start;
      }
    }
    LaneRec r;
    r.lo = lo_u;
    r.hi = hi_u;
    r.start = start_u;
    r.tiles = (hi_u - lo_u + tile - 1) / tile;
    r.item_begin = 0;
    r.n_items = 0;
    r.tmp_begin = 0;
    r.pad = 0;
    for (int m = 0; m < gang; ++m) lanes[l0 + m * lanes_per_unit] = r;
    my_tiles += r.tiles;
  }
  Scan2 tot;
  Scan2 pre = block_exclusive_scan2(Scan2{my_tiles, 0}, &tot);
  const long long T = tot.a;
  // With fewer tiles than CTAs only the first T CTAs get work, so that no
  // CTA's run is empty and every item covers at least one tile.
  const long long S = T < n_ctas ? (T > 0 ? T : 1) : n_ctas;

  // pass 2: items per work unit (number of CTA runs it overlaps)
  long long p = pre.a, my_items = 0, my_split = 0;
  for (int x = x0; x < x1; ++x) {
    const int l = lane_at(x);
    const int t = lanes[l].tiles;
    int n = 0;
    if (t > 0) n = cta_of(p + t - 1, T, S) - cta_of(p, T, S) + 1;
    for (int m = 0; m < gang; ++m) lanes[l + m * lanes_per_unit].n_items = n;
    lanes[l].pad = (int)p;  // tile prefix, used below and in pass 3
    my_items += n;
    if (n > 1) my_split += (long long)n * gang;
    p += t;
  }
  Scan2 tot2;
  Scan2 pre2 = block_exclusive_scan2(Scan2{my_items, my_split}, &tot2);

  if (group_order) {
    // row groups: the CTA runs their tiles span, and workspace rows for the
    // pieces of those that span several (the scans' barriers order these
    // reads of the tile prefixes after pass 2 and before pass 3)
    const int n_groups = rs.B;
    const int gper = (n_groups + kPlanThreads - 1) / kPlanThreads;
    const int g0 = threadIdx.x * gper, g1 = min(n_groups, g0 + gper);
    auto span = [&](int r, int* first) {
      const long long a = lanes[lane_at(r * group_lanes)].pad;
      const long long e = r + 1 < n_groups ? (long long)lanes[lane_at((r + 1) * group_lanes)].pad : T;
      *first = e > a ? cta_of(a, T, S) : 0;
      return e > a ? cta_of(e - 1, T, S) - *first + 1 : 0;
    };
    auto finished_apart = [](int n) { return n == 0 || n > kMlaMergeInKernel; };
    long long my_rows = 0, my_fin = 0;
    for (int r = g0; r < g1; ++r) {
      int first;
      const int n = span(r, &first);
      if (n > 1) my_rows += n;
      if (finished_apart(n)) ++my_fin;
    }
    Scan2 tot3;
    Scan2 pre3 = block_exclusive_scan2(Scan2{my_rows, my_fin}, &tot3);
    long long row = pre3.a, fin = pre3.b;
    for (int r = g0; r < g1; ++r) {
      GroupRec gr;
      gr.pieces = span(r, &gr.first_cta);
      gr.tmp_begin = gr.pieces > 1 ? (int)row : 0;
      gr.pad = 0;
      gr.cnt[0] = gr.cnt[1] = 0;
      gr.pad2[0] = gr.pad2[1] = 0;
      groups[r] = gr;
      if (gr.pieces > 1) row += gr.pieces;
      if (finished_apart(gr.pieces)) finish[fin++] = r;
    }
    n_finish = tot3.b;
    __syncthreads();
  }

  // pass 3: items (a gang's items name its first lane; lane m of the gang
  // keeps its split pieces in workspace rows tmp_begin + m * n_items ..)
  long long ib = pre2.a, tb = pre2.b;
  for (int x = x0; x < x1; ++x) {
    const int l = lane_at(x);
    LaneRec r = lanes[l];
    const long long P = r.pad;
    r.item_begin = (int)ib;
    r.pad = 0;
    for (int m = 0; m < gang; ++m) {
      r.tmp_begin = (int)(tb + (long long)m * r.n_items);
      lanes[l + m * lanes_per_unit] = r;
    }
    if (r.n_items > 0) {
      const int c0 = cta_of(P, T, S);
      for (int j = 0; j < r.n_items; ++j) {
        const int c = c0 + j;
        const long long cs = cta_start(c, T, S), ce = cta_start(c + 1, T, S);
        const long long a = cs > P ? cs : P;
        const long long e = ce < P + r.tiles ? ce : P + r.tiles;
        ItemRec it;
        it.lane = l;
        it.t0 = (int)(a - P);
        it.t1 = (int)(e - P);
        it.out_row = r.n_items > 1 ? (int)(tb + j) : -1;
        items[ib + j] = it;
        if (a == cs) cta_begin[c] = (int)(ib + j);  // first item of CTA c
      }
    }
    ib += r.n_items;
    if (r.n_items > 1) tb += (long long)r.n_items * gang;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int n_items = (int)tot2.a;
    // CTAs past the last run (T < n_ctas, or no tiles at all) get no items
    for (int c = (T > 0 ? (int)S : 0); c <= n_ctas; ++c) cta_begin[c] = n_items;
    hdr->n_items = n_items;
    hdr->n_lanes = n_lanes;
    hdr->n_ctas = n_ctas;
    hdr->total_tiles = (int)T;
    hdr->n_finish = (int)n_finish;
  }
}

}  // namespace

cudaError_t launch_plan(const RangeSpec& rs, int lanes_per_unit, int tile, int n_ctas, void* ws,
                        const WsLayout& L, bool group_order, int gang, cudaStream_t st) {
  plan_kernel<<<1, kPlanThreads, 0, st>>>(rs, lanes_per_unit, tile, n_ctas, static_cast<char*>(ws), L,
                                          group_order ? 1 : 0, gang);
  return cudaGetLastError();
}

}  // namespace dcp
