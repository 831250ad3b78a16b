// Internal declarations shared by the libdcp translation units.
//
// Work decomposition (all kernels): a *lane* is one independent softmax
// problem over a token range -- (shard, sequence, KV head, head group) for GQA,
// (shard, sequence) for MLA. Lanes are cut into tiles of TILE tokens. The
// plan kernel lays every lane's tiles end to end and gives each persistent
// CTA (or CTA pair) an equal, contiguous run of tiles, so work is balanced to
// one tile whatever the length mix. A CTA's run crosses at most a few lane
// boundaries; each piece of a lane it touches is an *item*. A lane covered by
// one item is written straight to the shard's partial output; a lane split
// over several items is written as per-item partials to the workspace and
// merged by the combine kernel (same LSE merge as across shards).
//
// MLA lays the lanes out row group by row group instead -- the N shard lanes
// of a query row next to each other -- so consecutive items of a CTA pair
// share their query. Its one-call path (partial attention and merge together)
// then carries one online softmax through the consecutive shards of a row
// group, so the shards are merged on chip: a row group whose tiles one CTA run
// covers is written straight to the output; one that a CTA boundary cuts
// leaves one *piece* per run in the workspace. Up to kMlaMergeInKernel pieces
// the CTA that writes the last piece merges them; a group cut into more (a
// few long sequences over many CTA runs, whose merges would all fall at the
// end of the kernel on a few SMs) and groups without tokens are finished by a
// short kernel over the whole GPU, from a list the plan writes.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dcp.h"

namespace dcp {

constexpr int kMaxShards = DCP_MAX_SHARDS;

// Shard descriptors passed by value as a kernel parameter.
struct ShardSet {
  const void* k[kMaxShards];
  const void* v[kMaxShards];
  const int32_t* table[kMaxShards];
  int64_t nblk[kMaxShards];
  int32_t max_blocks[kMaxShards];
};

// How a lane's token range is found: unit u = shard * B + r, where row group
// r = b * G + k holds query tokens [k*tpr, min(qlen, (k+1)*tpr)) of sequence
// b (G = ceil(qlen / tpr); one-token decode: r = b). Query token j attends
// positions below its causal limit lim_j = seq_lens[b] - (qlen - 1 - j); the
// group's range is clipped to the limit of its last token (a kernel masks
// each token at its own limit):
//   mode 0 (all shards): [starts[b*N+i], i<N-1 ? starts[b*N+i+1] : inf) clipped to lim
//   mode 1 (one shard) : [range[2b], range[2b+1]) clipped to lim
struct RangeSpec {
  const int32_t* seq_lens;
  const int32_t* starts;  // mode 0
  const int32_t* range;   // mode 1
  int32_t* err;           // device error flags (may be NULL)
  int mode;
  int B;                  // row groups per shard: sequences x G
  int N;
  int qlen;               // query tokens per sequence
  int tpr;                // query tokens per row group
};

struct LaneRec {     // 32 bytes
  int lo;            // first global position attended
  int hi;            // one past the last
  int start;         // global position of local position 0 (shard start)
  int tiles;         // ceil((hi - lo) / TILE)
  int item_begin;
  int n_items;
  int tmp_begin;     // first workspace partial row if n_items > 1
  int pad;
};

struct ItemRec {     // 16 bytes
  int lane;
  int t0;            // tile range [t0, t1) within the lane
  int t1;
  int out_row;       // >= 0: workspace partial row; -1: write the lane's output directly
};

constexpr int kMlaMergeInKernel = 4;  // pieces a group may have for the attention kernel to merge it

struct GroupRec {    // 32 bytes: one query row group of the one-call MLA path
  int pieces;        // CTA runs its tiles span (0: no tokens in any shard)
  int tmp_begin;     // first workspace partial row if pieces > 1
  int first_cta;     // CTA run of piece 0
  int pad;
  int cnt[2];        // pieces written, per CTA of the pair (zeroed by the plan)
  int pad2[2];
};

struct WsHeader {
  int n_items;
  int n_lanes;
  int n_ctas;
  int total_tiles;
  int n_finish;      // group order: row groups in the finish list
  int pad[59];       // 256 bytes
};

struct WsLayout {
  size_t lanes_off, items_off, cta_off, grp_off, fin_off, tmp_o_off, tmp_lse_off, total;
  int max_lanes, max_items, max_ctas, max_tmp, rows_per_lane, max_groups;
};

// Workspace layout for n_lanes lanes, up to max_ctas work CTAs, rows_per_lane
// query heads per lane, dv-wide outputs and n_groups group records (the row
// groups of the one-call MLA path; 0 where unused).
WsLayout ws_layout(int n_lanes, int max_ctas, int rows_per_lane, int dv, int n_groups);

// Per-device launch facts (cached).
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
};
int device_info(DeviceInfo* out);

// Lane geometry of a descriptor.
struct LaneGeom {
  int heads_per_lane;  // query heads of one lane
  int groups;          // lanes per (unit, kv head) for GQA (g > 16 -> several)
  int lanes_per_unit;  // kv_heads * groups (GQA) or 1 (MLA)
  int tile;            // tokens per tile
};
LaneGeom lane_geom(const dcp_attn_desc& d);

// Kernel launchers (return the launch's cudaError_t).
// group_order: lay the lanes out row group by row group, fill the group
// records and the finish list (MLA); otherwise shard by shard. gang > 1 (the
// many-row GQA kernel; gang divides the token groups per sequence): n_ctas
// counts gangs of `gang` CTAs, and a work unit is `gang` lanes of
// consecutive token groups of one (shard, sequence, KV head) over the union
// of their ranges, each CTA of the gang taking one lane.
cudaError_t launch_plan(const RangeSpec& rs, int lanes_per_unit, int tile, int n_ctas,
                        void* ws, const WsLayout& L, bool group_order, int gang, cudaStream_t st);
cudaError_t launch_gqa(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                       float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas,
                       int32_t* err, cudaStream_t st);
// Query tokens that share each K/V tile in the GQA kernel (1, 2 or 4).
int gqa_team(int qlen);
int gqa_ctas(const dcp_attn_desc& d, const DeviceInfo& di, int team);
// o non-NULL: the one-call path (plan laid out with group_order): the
// merged rows go to o / lse_out (NULL allowed) and o_parts / lses are unused.
cudaError_t launch_mla(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                       float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas,
                       int32_t* err, cudaStream_t st, float* o = nullptr, float* lse_out = nullptr);
int mla_ctas(const dcp_attn_desc& d, const DeviceInfo& di);
// Many query rows per KV head (GQA, head dim 128, bf16 cache, q_len * g >= 48):
// 128-row lanes of 128/g tokens x g heads on the tcgen05 tensor cores.
bool gqa_tc_eligible(const dcp_attn_desc& d, int qlen);
int gqa_tc_rows_tokens(const dcp_attn_desc& d, int qlen);  // query tokens per lane: 128 or 256 rows / g
int gqa_tc_ctas(const dcp_attn_desc& d, const DeviceInfo& di, int qlen);
// gang: CTAs per gang of the plan (n_ctas CTAs, n_ctas / gang gangs).
int gqa_tc_gang(int token_groups, int n_ctas);
cudaError_t launch_gqa_tc(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                          float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas, int gang,
                          int32_t* err, cudaStream_t st);
cudaError_t launch_combine(const dcp_attn_desc& d, const LaneGeom& lg, const RangeSpec& rs, int n_lanes,
                           const void* ws, const WsLayout& L, float* o_parts, float* lses, cudaStream_t st);
// Steps 2 and 3 joined: merges every output row's pieces across the shards
// (direct partial rows and split pieces in the workspace) into o / lse_out.
cudaError_t launch_combine_merge(const dcp_attn_desc& d, const LaneGeom& lg, const RangeSpec& rs, const void* ws,
                                 const WsLayout& L, const float* o_parts, const float* lses, float* o,
                                 float* lse_out, cudaStream_t st);
cudaError_t launch_merge(const float* o_parts, const float* lses, int N, int rows, int dv, float* o,
                         float* lse_out, cudaStream_t st);
cudaError_t launch_append(const dcp_attn_desc& d, const ShardSet& sh, int N, const int32_t* starts,
                          int B, const int32_t* seq_ids, const int32_t* positions, const void* k_new,
                          const void* v_new, int T, int32_t* err, cudaStream_t st);

// Device helpers ------------------------------------------------------------
__device__ __forceinline__ void raise_flag(int32_t* err, int bit) {
  if (err) atomicOr(err, bit);
}

}  // namespace dcp
