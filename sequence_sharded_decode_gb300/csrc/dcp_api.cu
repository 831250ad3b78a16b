// C ABI of libdcp: argument validation, routing plan, workspace sizing and
// the launch sequences of the three steps of decode context parallelism.
#include <cmath>
#include <cstring>
#include <mutex>

#include "dcp_internal.cuh"

namespace dcp {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int n_lanes, int max_ctas, int rows_per_lane, int dv, int n_groups) {
  WsLayout L;
  L.max_lanes = n_lanes;
  L.max_ctas = max_ctas;
  L.max_items = n_lanes + max_ctas;
  L.max_tmp = 2 * max_ctas;  // a lane cut k ways holds k-1 CTA boundaries, k <= 2(k-1)
  L.rows_per_lane = rows_per_lane;
  L.max_groups = n_groups;
  size_t off = sizeof(WsHeader);
  L.lanes_off = off;
  off = align256(off + sizeof(LaneRec) * (size_t)n_lanes);
  L.items_off = off;
  off = align256(off + sizeof(ItemRec) * (size_t)L.max_items);
  L.cta_off = off;
  off = align256(off + sizeof(int) * (size_t)(max_ctas + 1));
  L.grp_off = off;
  off = align256(off + sizeof(GroupRec) * (size_t)n_groups);
  L.fin_off = off;
  off = align256(off + sizeof(int) * (size_t)n_groups);
  L.tmp_o_off = off;
  off = align256(off + sizeof(float) * (size_t)L.max_tmp * rows_per_lane * dv);
  L.tmp_lse_off = off;
  off = align256(off + sizeof(float) * (size_t)L.max_tmp * rows_per_lane);
  L.total = off;
  return L;
}

int device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && have[dev]) {
    *out = cache[dev];
    return 0;
  }
  DeviceInfo di;
  if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return -1;
  if (dev < 64) {
    cache[dev] = di;
    have[dev] = true;
  }
  *out = di;
  return 0;
}

LaneGeom lane_geom(const dcp_attn_desc& d) {
  LaneGeom g;
  if (d.kind == DCP_KIND_MLA) {
    g.heads_per_lane = d.num_q_heads;
    g.groups = 1;
    g.lanes_per_unit = 1;
    g.tile = 64;
  } else {
    const int grp = d.num_q_heads / d.num_kv_heads;
    g.heads_per_lane = 16;
    g.groups = (grp + 15) / 16;
    g.lanes_per_unit = d.num_kv_heads * g.groups;
    g.tile = 16;
  }
  return g;
}

// Which kernel serves a step and how its lanes are cut.
//  MLA: one lane per (shard, query row), 128 head rows, 64-token tiles.
//  GQA, many rows per KV head (gqa_tc_eligible): one lane per (shard,
//    sequence, group of 128/g query tokens, KV head), 128 rows, 64-token
//    tiles, the tcgen05 kernel.
//  GQA otherwise: one lane per (shard, sequence, group of `team` query
//    tokens, KV head, group of up to 16 heads), 16-token tiles, the mma.sync
//    kernel whose team of warps shares each tile.
struct Path {
  LaneGeom lg;
  int tc;             // the tcgen05 GQA kernel
  int tpr;            // query tokens per row group
  int rows_per_lane;  // query rows of one lane
  int qlen;           // query tokens per sequence of the step
};
static Path path_for(const dcp_attn_desc& d, int q_len) {
  Path p;
  p.lg = lane_geom(d);
  p.tc = 0;
  p.qlen = q_len;
  if (d.kind == DCP_KIND_MLA) {
    p.tpr = 1;
    p.rows_per_lane = d.num_q_heads;
    return p;
  }
  const int grp = d.num_q_heads / d.num_kv_heads;
  if (gqa_tc_eligible(d, q_len)) {
    p.tc = 1;
    p.tpr = gqa_tc_rows_tokens(d, q_len);
    p.rows_per_lane = p.tpr * grp;
    p.lg.heads_per_lane = grp;
    p.lg.groups = 1;
    p.lg.lanes_per_unit = d.num_kv_heads;
    p.lg.tile = 64;
    return p;
  }
  p.tpr = gqa_team(q_len);
  p.rows_per_lane = (grp < 16 ? grp : 16) * p.tpr;
  return p;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_desc(const dcp_attn_desc* d) {
  if (!d) return DCP_ERR_INVALID_ARG;
  if (d->kind != DCP_KIND_GQA && d->kind != DCP_KIND_MLA) return DCP_ERR_INVALID_ARG;
  if (d->num_q_heads < 1 || d->num_kv_heads < 1 || d->head_dim_k < 1 || d->head_dim_v < 1 || d->block_size < 1)
    return DCP_ERR_SHAPE;
  if (d->num_q_heads % d->num_kv_heads) return DCP_ERR_SHAPE;
  if (!std::isfinite(d->scale)) return DCP_ERR_INVALID_ARG;
  if (d->kv_dtype != DCP_KV_BF16 && d->kv_dtype != DCP_KV_FP8_E4M3) return DCP_ERR_INVALID_ARG;
  if (d->kv_dtype == DCP_KV_FP8_E4M3) {
    if (!std::isfinite(d->k_scale) || !std::isfinite(d->v_scale) || !(d->k_scale > 0.f) || !(d->v_scale > 0.f))
      return DCP_ERR_INVALID_ARG;
  }
  if (d->kind == DCP_KIND_GQA) {
    if (d->head_dim_k != d->head_dim_v) return DCP_ERR_UNSUPPORTED;
    if (d->head_dim_k != 64 && d->head_dim_k != 128) return DCP_ERR_UNSUPPORTED;
    if (d->block_size % 16) return DCP_ERR_UNSUPPORTED;
    if (d->num_q_heads > 256) return DCP_ERR_UNSUPPORTED;
  } else {
    if (d->num_kv_heads != 1) return DCP_ERR_SHAPE;
    if (d->head_dim_v > d->head_dim_k) return DCP_ERR_SHAPE;
    if (d->head_dim_k != 576 || d->head_dim_v != 512 || d->num_q_heads != 128 || d->block_size != 64)
      return DCP_ERR_UNSUPPORTED;
  }
  return DCP_OK;
}

static int check_shards(const dcp_attn_desc& d, const dcp_shard* s, int N, ShardSet* out) {
  if (!s || N < 1 || N > kMaxShards) return DCP_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  for (int i = 0; i < N; ++i) {
    if (!s[i].k_pool || !s[i].block_table) return DCP_ERR_INVALID_ARG;
    if (d.kind == DCP_KIND_GQA && !s[i].v_pool) return DCP_ERR_INVALID_ARG;
    if (d.kind == DCP_KIND_MLA && s[i].v_pool) return DCP_ERR_INVALID_ARG;
    if (s[i].num_blocks < 1 || s[i].max_blocks_per_seq < 1) return DCP_ERR_SHAPE;
    if (!aligned16(s[i].k_pool) || (s[i].v_pool && !aligned16(s[i].v_pool))) return DCP_ERR_INVALID_ARG;
    out->k[i] = s[i].k_pool;
    out->v[i] = s[i].v_pool;
    out->table[i] = s[i].block_table;
    out->nblk[i] = s[i].num_blocks;
    out->max_blocks[i] = s[i].max_blocks_per_seq;
  }
  return DCP_OK;
}

static int work_ctas(const dcp_attn_desc& d, const DeviceInfo& di, const Path& p) {
  if (d.kind == DCP_KIND_MLA) return mla_ctas(d, di);
  return p.tc ? gqa_tc_ctas(d, di, p.qlen) : gqa_ctas(d, di, p.tpr);
}

// Workspace layout for B row groups per shard (sequences x token groups).
static int layout_for(const dcp_attn_desc& d, int B, int N, const Path& p, WsLayout* L, int* n_ctas) {
  DeviceInfo di;
  if (device_info(&di) != 0) return DCP_ERR_CUDA;
  const int c = work_ctas(d, di, p);
  if (c <= 0) return DCP_ERR_CUDA;
  const long long lanes = (long long)B * N * p.lg.lanes_per_unit;
  if (lanes > (1 << 26)) return DCP_ERR_SHAPE;
  *L = ws_layout((int)lanes, c, p.rows_per_lane, d.head_dim_v, d.kind == DCP_KIND_MLA ? B : 0);
  *n_ctas = c;
  return DCP_OK;
}

// Plan, attention kernel, then either the combine of split lanes into the
// shards' partial rows, or (o non-NULL) the one-pass merge of every output
// row across shards and split pieces into o / lse_out.
static int run_partial(const dcp_attn_desc* desc, const Path& path, const void* q, const ShardSet& sh,
                       const RangeSpec& rs, float* o_parts, float* lses, void* ws, size_t ws_bytes, int32_t* err,
                       void* stream, float* o = nullptr, float* lse_out = nullptr) {
  const dcp_attn_desc& d = *desc;
  WsLayout L;
  int n_ctas = 0;
  int rc = layout_for(d, rs.B, rs.N, path, &L, &n_ctas);
  if (rc != DCP_OK) return rc;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return DCP_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const LaneGeom& g = path.lg;
  // MLA with o: the attention kernel merges the shards itself
  const bool mla_merge = d.kind == DCP_KIND_MLA && o != nullptr;
  // many-row GQA: gangs of CTAs over the token groups of one KV range
  const int gang = path.tc ? gqa_tc_gang((rs.qlen + rs.tpr - 1) / rs.tpr, n_ctas) : 1;
  if (launch_plan(rs, g.lanes_per_unit, g.tile, n_ctas / gang, ws, L, d.kind == DCP_KIND_MLA, gang, st) !=
      cudaSuccess)
    return DCP_ERR_CUDA;
  cudaError_t e;
  if (d.kind == DCP_KIND_MLA)
    e = launch_mla(d, q, sh, rs, o_parts, lses, ws, L, n_ctas, err, st, mla_merge ? o : nullptr, lse_out);
  else if (path.tc) e = launch_gqa_tc(d, q, sh, rs, o_parts, lses, ws, L, n_ctas, gang, err, st);
  else e = launch_gqa(d, q, sh, rs, o_parts, lses, ws, L, n_ctas, err, st);
  if (e == cudaErrorNotSupported) return DCP_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return DCP_ERR_CUDA;
  if (mla_merge) {
    // nothing left: the rows are merged
  } else if (o) {
    if (launch_combine_merge(d, g, rs, ws, L, o_parts, lses, o, lse_out, st) != cudaSuccess) return DCP_ERR_CUDA;
  } else if (launch_combine(d, g, rs, L.max_lanes, ws, L, o_parts, lses, st) != cudaSuccess) {
    return DCP_ERR_CUDA;
  }
  return DCP_OK;
}

// Fixed scratch of dcp_decode_partial_all_noalloc: the library's own device
// array, for callers that cannot allocate. Host code must not pass the
// symbol itself to a kernel (in host code it names a host-side stand-in);
// noalloc_scratch() looks up its device address once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DCP_NOALLOC_SCRATCH_BYTES];

static int noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DCP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DCP_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return DCP_OK;
}

}  // namespace dcp

using namespace dcp;

extern "C" {

const char* dcp_status_string(int status) {
  switch (status) {
    case DCP_OK: return "ok";
    case DCP_ERR_INVALID_ARG: return "invalid argument";
    case DCP_ERR_SHAPE: return "inconsistent shape";
    case DCP_ERR_UNSUPPORTED: return "unsupported configuration";
    case DCP_ERR_CUDA: return "CUDA error";
    case DCP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DCP_ERR_SCRATCH_LIMIT:
      return "problem needs more workspace than the fixed scratch of dcp_decode_partial_all_noalloc";
    default: return "unknown status";
  }
}

int dcp_version(void) { return 400; }

int dcp_shard_plan(const int32_t* ctx_lens, int B, int N, int block_size, int reserve_tokens,
                   int32_t* shard_starts, int32_t* blocks_needed) {
  if (B < 0 || N < 1 || N > DCP_MAX_SHARDS || block_size < 1 || reserve_tokens < 0) return DCP_ERR_INVALID_ARG;
  if (B > 0 && (!ctx_lens || !shard_starts)) return DCP_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const long long L0 = ctx_lens[b];
    if (L0 < 0) return DCP_ERR_INVALID_ARG;
    long long C = (L0 + N - 1) / N;
    if (C < 1) C = 1;
    const long long end = L0 + reserve_tokens;
    if ((long long)(N - 1) * C > INT32_MAX || end > INT32_MAX) return DCP_ERR_INVALID_ARG;
    for (int i = 0; i < N; ++i) {
      const long long lo = (long long)i * C;
      shard_starts[(size_t)b * N + i] = (int32_t)lo;
      if (blocks_needed) {
        long long hi = (i == N - 1) ? end : (lo + C < end ? lo + C : end);
        const long long tokens = hi > lo ? hi - lo : 0;
        blocks_needed[(size_t)b * N + i] = (int32_t)((tokens + block_size - 1) / block_size);
      }
    }
  }
  return DCP_OK;
}

int dcp_kv_append(const dcp_attn_desc* desc, const dcp_shard* shards, int N, const int32_t* shard_starts, int B,
                  const int32_t* seq_ids, const int32_t* positions, const void* k_new, const void* v_new, int T,
                  int32_t* dev_err_flag, void* stream) {
  int rc = check_desc(desc);
  if (rc != DCP_OK) return rc;
  ShardSet sh;
  rc = check_shards(*desc, shards, N, &sh);
  if (rc != DCP_OK) return rc;
  if (T < 0 || B < 0) return DCP_ERR_INVALID_ARG;
  if (!seq_ids && T != B) return DCP_ERR_SHAPE;
  if (T == 0) return DCP_OK;
  if (!shard_starts || !positions || !k_new) return DCP_ERR_INVALID_ARG;
  if (desc->kind == DCP_KIND_GQA && !v_new) return DCP_ERR_INVALID_ARG;
  if (desc->kind == DCP_KIND_MLA && v_new) return DCP_ERR_INVALID_ARG;
  if (!aligned16(k_new) || (v_new && !aligned16(v_new))) return DCP_ERR_INVALID_ARG;
  if (launch_append(*desc, sh, N, shard_starts, B, seq_ids, positions, k_new, v_new, T, dev_err_flag,
                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DCP_ERR_CUDA;
  return DCP_OK;
}

size_t dcp_workspace_size(const dcp_attn_desc* desc, int B, int N) {
  return dcp_workspace_size_mtp(desc, B, 1, N);
}

size_t dcp_workspace_size_mtp(const dcp_attn_desc* desc, int B, int q_len, int N) {
  if (check_desc(desc) != DCP_OK || B < 0 || N < 1 || N > DCP_MAX_SHARDS) return 0;
  if (q_len < 1 || q_len > DCP_MAX_QUERY_TOKENS) return 0;
  const Path path = path_for(*desc, q_len);
  const long long rows = (long long)B * ((q_len + path.tpr - 1) / path.tpr);
  if (rows > INT32_MAX) return 0;
  WsLayout L;
  int n_ctas = 0;
  if (layout_for(*desc, (int)rows, N, path, &L, &n_ctas) != DCP_OK) return 0;
  return L.total;
}

int dcp_decode_partial(const dcp_attn_desc* desc, const void* q, const dcp_shard* shard, const int32_t* seq_lens,
                       const int32_t* shard_range, int B, float* o_part, float* lse, void* workspace,
                       size_t ws_bytes, int32_t* dev_err_flag, void* stream) {
  int rc = check_desc(desc);
  if (rc != DCP_OK) return rc;
  ShardSet sh;
  rc = check_shards(*desc, shard, 1, &sh);
  if (rc != DCP_OK) return rc;
  if (B < 0) return DCP_ERR_INVALID_ARG;
  if (B == 0) return DCP_OK;
  if (!q || !seq_lens || !shard_range || !o_part || !lse) return DCP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o_part)) return DCP_ERR_INVALID_ARG;
  RangeSpec rs{seq_lens, nullptr, shard_range, dev_err_flag, 1, B, 1, 1, 1};
  return run_partial(desc, path_for(*desc, 1), q, sh, rs, o_part, lse, workspace, ws_bytes, dev_err_flag, stream);
}

int dcp_decode_partial_all(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards, int N,
                           const int32_t* seq_lens, const int32_t* shard_starts, int B, float* o_parts, float* lses,
                           void* workspace, size_t ws_bytes, int32_t* dev_err_flag, void* stream) {
  return dcp_decode_partial_all_mtp(desc, q, shards, N, seq_lens, shard_starts, B, 1, o_parts, lses, workspace,
                                    ws_bytes, dev_err_flag, stream);
}

int dcp_decode_partial_all_mtp(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards, int N,
                               const int32_t* seq_lens, const int32_t* shard_starts, int B, int q_len,
                               float* o_parts, float* lses, void* workspace, size_t ws_bytes,
                               int32_t* dev_err_flag, void* stream) {
  int rc = check_desc(desc);
  if (rc != DCP_OK) return rc;
  ShardSet sh;
  rc = check_shards(*desc, shards, N, &sh);
  if (rc != DCP_OK) return rc;
  if (B < 0 || q_len < 1 || q_len > DCP_MAX_QUERY_TOKENS) return DCP_ERR_INVALID_ARG;
  if (B == 0) return DCP_OK;
  if (!q || !seq_lens || !shard_starts || !o_parts || !lses) return DCP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o_parts)) return DCP_ERR_INVALID_ARG;
  if ((long long)B * q_len > INT32_MAX) return DCP_ERR_SHAPE;
  const Path path = path_for(*desc, q_len);
  const long long groups = (q_len + path.tpr - 1) / path.tpr;
  if ((long long)B * groups > INT32_MAX) return DCP_ERR_SHAPE;
  RangeSpec rs{seq_lens, shard_starts, nullptr, dev_err_flag, 0, (int)(B * groups), N, q_len, path.tpr};
  return run_partial(desc, path, q, sh, rs, o_parts, lses, workspace, ws_bytes, dev_err_flag, stream);
}

int dcp_attention_all(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards, int N,
                      const int32_t* seq_lens, const int32_t* shard_starts, int B, int q_len, float* o_parts,
                      float* lses, float* o, float* lse_out, void* workspace, size_t ws_bytes,
                      int32_t* dev_err_flag, void* stream) {
  int rc = check_desc(desc);
  if (rc != DCP_OK) return rc;
  ShardSet sh;
  rc = check_shards(*desc, shards, N, &sh);
  if (rc != DCP_OK) return rc;
  if (B < 0 || q_len < 1 || q_len > DCP_MAX_QUERY_TOKENS) return DCP_ERR_INVALID_ARG;
  if (B == 0) return DCP_OK;
  if (!q || !seq_lens || !shard_starts || !o_parts || !lses || !o) return DCP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o_parts) || !aligned16(o)) return DCP_ERR_INVALID_ARG;
  if (desc->head_dim_v % 4 || desc->head_dim_v > 512) return DCP_ERR_UNSUPPORTED;
  if ((long long)B * q_len > INT32_MAX) return DCP_ERR_SHAPE;
  const Path path = path_for(*desc, q_len);
  const long long groups = (q_len + path.tpr - 1) / path.tpr;
  if ((long long)B * groups > INT32_MAX) return DCP_ERR_SHAPE;
  RangeSpec rs{seq_lens, shard_starts, nullptr, dev_err_flag, 0, (int)(B * groups), N, q_len, path.tpr};
  return run_partial(desc, path, q, sh, rs, o_parts, lses, workspace, ws_bytes, dev_err_flag, stream, o, lse_out);
}

int dcp_decode_partial_all_noalloc(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards, int N,
                                   const int32_t* seq_lens, const int32_t* shard_starts, int B, float* o_parts,
                                   float* lses, int32_t* dev_err_flag, void* stream) {
  int rc = check_desc(desc);
  if (rc != DCP_OK) return rc;
  ShardSet sh;
  rc = check_shards(*desc, shards, N, &sh);
  if (rc != DCP_OK) return rc;
  if (B < 0) return DCP_ERR_INVALID_ARG;
  if (B == 0) return DCP_OK;
  if (!q || !seq_lens || !shard_starts || !o_parts || !lses) return DCP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o_parts)) return DCP_ERR_INVALID_ARG;
  WsLayout L;
  int n_ctas = 0;
  const Path path = path_for(*desc, 1);
  rc = layout_for(*desc, B, N, path, &L, &n_ctas);
  if (rc != DCP_OK) return rc;
  if (L.total > DCP_NOALLOC_SCRATCH_BYTES) return DCP_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  rc = noalloc_scratch(&ws);
  if (rc != DCP_OK) return rc;
  RangeSpec rs{seq_lens, shard_starts, nullptr, dev_err_flag, 0, B, N, 1, 1};
  return run_partial(desc, path, q, sh, rs, o_parts, lses, ws, DCP_NOALLOC_SCRATCH_BYTES, dev_err_flag, stream);
}

int dcp_merge(const float* o_parts, const float* lses, int N, int B, int Hq, int Dv, float* o, float* lse_out,
              void* stream) {
  if (N < 1 || B < 0 || Hq < 1 || Dv < 1) return DCP_ERR_INVALID_ARG;
  if (Dv % 4) return DCP_ERR_UNSUPPORTED;
  if (B == 0) return DCP_OK;
  if (!o_parts || !lses || !o) return DCP_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o)) return DCP_ERR_INVALID_ARG;
  const long long rows = (long long)B * Hq;
  if (rows > INT32_MAX) return DCP_ERR_SHAPE;
  if (launch_merge(o_parts, lses, N, (int)rows, Dv, o, lse_out, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DCP_ERR_CUDA;
  return DCP_OK;
}

}  // extern "C"
