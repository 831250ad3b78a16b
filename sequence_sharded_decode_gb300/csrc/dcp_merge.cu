// LSE merge of partial attention results (step 3 of the method: the partial
// outputs of the shards are combined by online-softmax reweighting into the
// exact full-context attention -- Qiita write-up "vLLMの-dcpが長文脈のKV
// キャッシュ重複を消して3倍速くする", section "トークンの区間でGPUに割り振る";
// "Inference Systems Infrastructure Notes (7): DCP", sections 2-3).
//
// For every output row r (a (sequence, query head) pair) and partials i:
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   O = sum_i w_i O_i / sum_i w_i,  lse = M + ln sum_i w_i,
// an all-empty row (every lse_i = -inf) gives O = 0, lse = -inf.
//
// The same arithmetic serves two places: dcp_merge combines the N shard
// partials held in the caller's scratch buffer, and the combine kernel joins
// the pieces of a lane that the balanced split cut across several CTAs. Both
// stream fp32 rows with 16-byte loads: HBM-bound.
#include <cmath>

#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr int kMergeThreads = 256;

// One warp per row: lane i < N reads lse_i; the weights are broadcast by
// shuffles; the row's Dv/4 float4 columns are spread over the lanes.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ o_parts,
                                                              const float* __restrict__ lses, int N,
                                                              long long rows, int dv4, float* __restrict__ o,
                                                              float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (kMergeThreads / 32);
  for (long long r = (long long)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
    float M = -INFINITY;
    for (int i = lane; i < N; i += 32) M = fmaxf(M, lses[(long long)i * rows + r]);
    for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    const float4* src = reinterpret_cast<const float4*>(o_parts);
    float4* dst = reinterpret_cast<float4*>(o) + r * dv4;
    if (M == -INFINITY) {
      for (int c = lane; c < dv4; c += 32) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lse_out && lane == 0) lse_out[r] = -INFINITY;
      continue;
    }
    float wsum = 0.f;
    for (int i = lane; i < N; i += 32) {
      const float li = lses[(long long)i * rows + r];
      wsum += li == -INFINITY ? 0.f : expf(li - M);
    }
    for (int s = 16; s > 0; s >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, s);
    const float inv = 1.f / wsum;
    for (int c = lane; c < dv4; c += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < N; ++i) {
        const float li = lses[(long long)i * rows + r];
        if (li == -INFINITY) continue;
        const float w = expf(li - M);
        const float4 v = src[((long long)i * rows + r) * dv4 + c];
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      dst[c] = acc;
    }
    if (lse_out && lane == 0) lse_out[r] = M + logf(wsum);
  }
}

// Joins the items of split lanes (workspace partial rows) into the lane's
// output rows; writes O = 0, LSE = -inf for lanes with no tokens at all.
// One warp per (lane, query-head row), float4 columns spread over the lanes;
// warps of lanes written directly by the attention kernel return at once.
struct CombineGeom {
  int Hq, dv, lanes_per_unit, heads_per_lane, groups, g;
  int B;     // row groups per shard (sequences x token groups)
  int G;     // token groups per sequence
  int tpr;   // query tokens per row group
  int qlen;  // query tokens per sequence
};

__global__ void __launch_bounds__(kMergeThreads) combine_kernel(const char* __restrict__ ws, WsLayout L,
                                                                CombineGeom cg, float* __restrict__ o_parts,
                                                                float* __restrict__ lses) {
  const int Hq = cg.Hq, dv = cg.dv, groups = cg.groups;
  const int lane = threadIdx.x & 31;
  const int rpl = L.rows_per_lane;
  const long long total = (long long)L.max_lanes * rpl;
  const long long warps = (long long)gridDim.x * (kMergeThreads / 32);
  const LaneRec* lrec = reinterpret_cast<const LaneRec*>(ws + L.lanes_off);
  const float* tmp_o = reinterpret_cast<const float*>(ws + L.tmp_o_off);
  const float* tmp_lse = reinterpret_cast<const float*>(ws + L.tmp_lse_off);
  const int dv4 = dv / 4;
  for (long long w = (long long)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5); w < total; w += warps) {
    const int lane_id = (int)(w / rpl), r = (int)(w - (long long)lane_id * rpl);
    const LaneRec ln = lrec[lane_id];
    if (ln.n_items == 1) continue;
    const int u = lane_id / cg.lanes_per_unit, j = lane_id - u * cg.lanes_per_unit;
    int head0, nheads;
    if (groups > 0) {  // GQA lane = (unit, kv head, head group)
      const int kvh = j / groups, hg = j - kvh * groups;
      head0 = kvh * cg.g + hg * cg.heads_per_lane;
      nheads = min(cg.heads_per_lane, cg.g - hg * cg.heads_per_lane);
    } else {
      head0 = 0;
      nheads = Hq;
    }
    // row r of the lane = (query token slot js of the row group, head hr)
    const int rpt = rpl / cg.tpr;
    const int js = r / rpt, hr = r - js * rpt;
    const int shard = u / cg.B, rg = u - shard * cg.B;
    const int b = rg / cg.G, jt = (rg - b * cg.G) * cg.tpr + js;
    if (hr >= nheads || jt >= cg.qlen) continue;
    const size_t orow = ((size_t)shard * (cg.B / cg.G) * cg.qlen + (size_t)b * cg.qlen + jt) * Hq + head0 + hr;
    float4* dst = reinterpret_cast<float4*>(o_parts + orow * dv);
    float* dst_lse = lses + orow;
    const int n = ln.n_items;
    float M = -INFINITY;
    for (int i = lane; i < n; i += 32) M = fmaxf(M, tmp_lse[(size_t)(ln.tmp_begin + i) * rpl + r]);
    for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    if (M == -INFINITY) {  // no tokens (or no items) for this lane
      for (int c = lane; c < dv4; c += 32) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) *dst_lse = -INFINITY;
      continue;
    }
    float wsum = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float li = tmp_lse[(size_t)(ln.tmp_begin + i) * rpl + r];
      wsum += li == -INFINITY ? 0.f : expf(li - M);
    }
    for (int s = 16; s > 0; s >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, s);
    const float inv = 1.f / wsum;
    for (int c = lane; c < dv4; c += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < n; ++i) {
        const size_t row = (size_t)(ln.tmp_begin + i) * rpl + r;
        const float li = tmp_lse[row];
        if (li == -INFINITY) continue;
        const float wt = expf(li - M);
        const float4 v = reinterpret_cast<const float4*>(tmp_o + row * dv)[c];
        acc.x += wt * v.x;
        acc.y += wt * v.y;
        acc.z += wt * v.z;
        acc.w += wt * v.w;
      }
      dst[c] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (lane == 0) *dst_lse = M + logf(wsum);
  }
}

// Steps 2 and 3 joined after the attention kernel: every output row
// (sequence, query token, head) merges, in one pass, the pieces of all N
// shards -- a shard's partial row where one item covered its lane, its
// split pieces in the workspace otherwise (none for an empty lane). One warp
// per row; the pieces' LSEs are read by every lane (broadcast), the row's
// float4 columns are spread over the lanes.
__global__ void __launch_bounds__(kMergeThreads) combine_merge_kernel(const char* __restrict__ ws, WsLayout L,
                                                                      CombineGeom cg, int N,
                                                                      const float* __restrict__ o_parts,
                                                                      const float* __restrict__ lses,
                                                                      float* __restrict__ o,
                                                                      float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int rpl = L.rows_per_lane, rpt = rpl / cg.tpr, dv4 = cg.dv / 4;
  const long long rows = (long long)(cg.B / cg.G) * cg.qlen * cg.Hq;  // output rows (= partial rows of a shard)
  const long long warps = (long long)gridDim.x * (kMergeThreads / 32);
  const LaneRec* lrec = reinterpret_cast<const LaneRec*>(ws + L.lanes_off);
  const float* tmp_o = reinterpret_cast<const float*>(ws + L.tmp_o_off);
  const float* tmp_lse = reinterpret_cast<const float*>(ws + L.tmp_lse_off);
  for (long long ro = (long long)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5); ro < rows; ro += warps) {
    const int h = (int)(ro % cg.Hq);
    const long long t = ro / cg.Hq;  // b * qlen + jt
    const int b = (int)(t / cg.qlen), jt = (int)(t - (long long)b * cg.qlen);
    const int rg = b * cg.G + jt / cg.tpr, js = jt % cg.tpr;
    int j, hr;  // lane within the unit, head row within the lane
    if (cg.groups > 0) {
      const int kvh = h / cg.g, hg = (h - kvh * cg.g) / cg.heads_per_lane;
      j = kvh * cg.groups + hg;
      hr = h - (kvh * cg.g + hg * cg.heads_per_lane);
    } else {
      j = 0;
      hr = h;
    }
    const int R = js * rpt + hr;
    float M = -INFINITY;
    for (int i = 0; i < N; ++i) {
      const LaneRec ln = lrec[((long long)i * cg.B + rg) * cg.lanes_per_unit + j];
      if (ln.n_items == 1) {
        M = fmaxf(M, lses[(long long)i * rows + ro]);
      } else {
        for (int k = 0; k < ln.n_items; ++k) M = fmaxf(M, tmp_lse[(long long)(ln.tmp_begin + k) * rpl + R]);
      }
    }
    float4* dst = reinterpret_cast<float4*>(o) + ro * dv4;
    if (M == -INFINITY) {  // no tokens in any shard
      for (int c = lane; c < dv4; c += 32) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lse_out && lane == 0) lse_out[ro] = -INFINITY;
      continue;
    }
    // the columns of this lane (at most 4 float4 per lane: Dv <= 512)
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    auto add = [&](const float* row, float li) {
      if (li == -INFINITY) return;
      const float w = expf(li - M);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(row);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = lane + 32 * q;
        if (c < dv4) {
          const float4 v = src[c];
          acc[q].x += w * v.x;
          acc[q].y += w * v.y;
          acc[q].z += w * v.z;
          acc[q].w += w * v.w;
        }
      }
    };
    for (int i = 0; i < N; ++i) {
      const LaneRec ln = lrec[((long long)i * cg.B + rg) * cg.lanes_per_unit + j];
      if (ln.n_items == 1) {
        const long long pr = (long long)i * rows + ro;
        add(o_parts + pr * cg.dv, lses[pr]);
      } else {
        for (int k = 0; k < ln.n_items; ++k) {
          const long long pr = (long long)(ln.tmp_begin + k) * rpl + R;
          add(tmp_o + pr * cg.dv, tmp_lse[pr]);
        }
      }
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = lane + 32 * q;
      if (c < dv4) dst[c] = make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
    }
    if (lse_out && lane == 0) lse_out[ro] = M + logf(wsum);
  }
}

}  // namespace

cudaError_t launch_combine_merge(const dcp_attn_desc& d, const LaneGeom& lg, const RangeSpec& rs, const void* ws,
                                 const WsLayout& L, const float* o_parts, const float* lses, float* o,
                                 float* lse_out, cudaStream_t st) {
  if (d.head_dim_v % 4 || d.head_dim_v > 512) return cudaErrorInvalidValue;
  CombineGeom cg;
  cg.Hq = d.num_q_heads;
  cg.dv = d.head_dim_v;
  cg.lanes_per_unit = lg.lanes_per_unit;
  cg.heads_per_lane = lg.heads_per_lane;
  cg.groups = d.kind == DCP_KIND_GQA ? lg.groups : 0;
  cg.g = d.num_q_heads / d.num_kv_heads;
  cg.tpr = rs.tpr;
  cg.qlen = rs.qlen;
  cg.G = (rs.qlen + rs.tpr - 1) / rs.tpr;
  cg.B = rs.B;
  DeviceInfo di;
  if (device_info(&di) != 0) return cudaErrorUnknown;
  const long long rows = (long long)(rs.B / cg.G) * rs.qlen * d.num_q_heads;
  if (rows <= 0) return cudaSuccess;
  const long long want = (rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
  const int grid = (int)(want < di.sm_count * 16LL ? want : di.sm_count * 16LL);
  combine_merge_kernel<<<grid, kMergeThreads, 0, st>>>(static_cast<const char*>(ws), L, cg, rs.N, o_parts, lses, o,
                                                       lse_out);
  return cudaGetLastError();
}

cudaError_t launch_merge(const float* o_parts, const float* lses, int N, int rows, int dv, float* o,
                         float* lse_out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  DeviceInfo di;
  if (device_info(&di) != 0) return cudaErrorUnknown;
  const long long want = ((long long)rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
  const int grid = (int)(want < di.sm_count * 16LL ? want : di.sm_count * 16LL);
  merge_kernel<<<grid, kMergeThreads, 0, st>>>(o_parts, lses, N, rows, dv / 4, o, lse_out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const dcp_attn_desc& d, const LaneGeom& lg, const RangeSpec& rs, int n_lanes,
                           const void* ws, const WsLayout& L, float* o_parts, float* lses, cudaStream_t st) {
  if (n_lanes <= 0) return cudaSuccess;
  CombineGeom cg;
  cg.Hq = d.num_q_heads;
  cg.dv = d.head_dim_v;
  cg.lanes_per_unit = lg.lanes_per_unit;
  cg.heads_per_lane = lg.heads_per_lane;
  cg.groups = d.kind == DCP_KIND_GQA ? lg.groups : 0;
  cg.g = d.num_q_heads / d.num_kv_heads;
  cg.tpr = rs.tpr;
  cg.qlen = rs.qlen;
  cg.G = (rs.qlen + rs.tpr - 1) / rs.tpr;
  cg.B = rs.B;
  DeviceInfo di;
  if (device_info(&di) != 0) return cudaErrorUnknown;
  const long long warps = (long long)n_lanes * L.rows_per_lane;
  const long long want = (warps + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
  const int grid = (int)(want < di.sm_count * 16LL ? want : di.sm_count * 16LL);
  combine_kernel<<<grid, kMergeThreads, 0, st>>>(static_cast<const char*>(ws), L, cg, o_parts, lses);
  return cudaGetLastError();
}

}  // namespace dcp
