// Partial decode attention, MLA-absorbed form, on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA) of sm_103a.
//
// What it computes (step 2 of the method: each shard attends the one-token
// queries against its own KV slice and emits a partial output plus LSE --
// Qiita write-up "vLLMの-dcpが長文脈のKVキャッシュ重複を消して3倍速くする",
// section "トークンの区間でGPUに割り振る"): per sequence, 128 absorbed query
// heads (576 wide) attend one latent KV head; the key is the cached 576-wide
// latent row and the value its first 512 entries (MLA keeps effectively one KV
// head -- same write-up, section "なぜテンソル並列だとKVキャッシュが二重に載るのか").
//
// Two kernels. The bf16 cache runs mla_split_kernel (further below: each CTA of
// the pair scores its own half of each page's tokens and the pair exchanges row
// maxima and P through distributed shared memory, which frees enough shared
// memory for three pipeline stages). The 8-bit cache runs mla_partial_kernel,
// described here, in which the two CTAs repeat the score.
//
// Layout of the work: the fp32 output accumulator of 128 heads x 512 dims is
// 256 KB, all of one SM's tensor memory, so each work item runs on a 2-CTA
// cluster and CTA r accumulates output dims [256 r, 256 r + 256). In
// mla_partial_kernel the two CTAs share no data: each computes the full
// scores S = Q K^T of the tile itself (the score MMA is repeated).
// (A tcgen05 pair MMA does not avoid the repeat: the pair's two halves of an
// operand sit at the same shared-memory offsets in both CTAs, so a token half
// of the page for the score and a value-dim half for P.V cannot share bytes,
// and 128 heads fill only half of a pair MMA's 256 rows.) Both CTAs need
// every page; the pair copies each page once: each CTA fetches alternate
// 64-column boxes and the copy (TMA multicast) lands in both CTAs, so a
// stage is free again only when both CTAs' P.V of its page finished. CTA 0
// also pulls each page into L2 four pages ahead. Measured against each CTA
// copying the whole page itself: +5.8 % on the 512-sequence workload (half
// the L2 reads; it no longer runs into the power cap), -2 to -3 % on MLA long
// and MLA decode (the coupled stage release). Per 64-token tile (= one paged
// block):
//   1. S = Q . K^T (M=128 heads, N=64 tokens, K=576) into TMEM; query dims
//      0-383 are the MMA's A operand in TMEM, dims 384-575 in shared memory
//   2. online softmax per head row, in log2 units, lazy rescale of O (only
//      when the running max grows by more than 2^8): eight warps, two per
//      TMEM lane quadrant; both read all 64 scores of their rows and take the
//      same maximum, each exponentiates its own 32 tokens and keeps their
//      row sum; the two sums meet once per item, for the epilogue
//   3. P as two bf16 terms, hi = bf16(p) and lo = p - hi truncated to bf16
//      (split with integer operations: conversion instructions share the
//      SFU's issue slots with ex2), so P.V carries ~15 mantissa bits of p;
//      P is written into the tile's own stage, over the four boxes of the
//      other CTA's value dims (read only by the score MMA), so each stage
//      has its own P buffer
//   4. O_r += P_hi . V_r (M=128, N=256, K=64) into TMEM, plus P_lo . V_r for
//      tiles that carry more than 1/32 of some row's running weight (the
//      first tiles of an item, or a tile with a dominant token); for the
//      others, dropping the residual changes O by at most 2^-8 x (that
//      tile's share of the row weight, < 1/32) x max|v|, and the MMA is
//      skipped.
// TMA brings each page as nine 64-column, 128-byte-swizzled boxes into a
// 2-stage ring. Two warps issue MMAs, one for the scores and one for the P.V
// products, so that a P.V enters the tensor pipe as soon as its P is ready;
// both poll their barriers with the non-blocking test_wait (a suspended
// try_wait reacts hundreds of cycles late) and run with uniform control flow
// so that one elect.sync-chosen lane issues each MMA without per-instruction
// operand shuffling. Measured on this part (clock64 traces of MLA long), a
// page spends ~2,000-2,400 cycles in flight, ~1,450 in the score MMA, ~1,500
// in the softmax and P stores and ~600 in P.V, and a stage holds its page
// through all of it: with two 72 KB stages per CTA (all the shared memory the
// query tail leaves) the period is about half that chain. Every barrier's
// phases are observed in order and never more than one phase late, so parity
// waits are unambiguous; every wait is bounded: on expiry the kernel raises
// DCP_DEVERR_TIMEOUT, stops all roles, drains what it issued and frees TMEM.
//
// The plan lays each query row group's N shard lanes next to each other, so
// consecutive items of a CTA pair mostly share their query: it stays in place
// (and the next row group's query is pulled into L2 one item ahead).
//
// One-call path (o non-NULL; step 3 joined to step 2, "Inference Systems
// Infrastructure Notes (7): DCP", section 3: intermediate results stay in
// reused buffers -- here, on chip): a CTA pair whose run holds several shards
// of a row group carries one online softmax through them -- the running
// maximum, row sums and O simply continue from one shard's tiles to the next,
// which is the LSE reweighting of the merge done as it goes. A row group whose
// tiles lie in one CTA run is written to o directly; one cut by run
// boundaries leaves one normalised piece (and its LSE) per run in the
// workspace. Up to kMlaMergeInKernel pieces, each CTA counts its piece with an
// atomic and the CTA whose count completes the group merges the pieces of its
// value dims (the same reweighting) into o; groups cut into more pieces, and
// groups without tokens, are finished by mla_finish_kernel over the whole GPU.
// No CTA ever waits for another.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "dcp_internal.cuh"
#include "dcp_tc_ptx.cuh"

namespace dcp {
namespace {

constexpr int kHeads = 128;
constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kTile = 64;                        // tokens per tile: one paged block
constexpr int kChunks = 9;                       // 64-column boxes per page (576 columns)
constexpr int kKStepsTmem = 24;                  // query dims 0-383: A operand in TMEM
constexpr int kKSteps = 36;                      // 16-column k-steps of the score MMA
constexpr int kQSmemChunks = 3;                  // query dims 384-575 in shared memory
constexpr int kStages = 2;                       // K/V tile pipeline depth
constexpr int kSoftmaxWarps = 8;                 // two per TMEM lane quadrant: token / value-dim halves
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;   // score MMAs (and the TMEM allocation)
constexpr int kPvWarp = kSoftmaxWarps + 2;    // P.V MMAs
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr int kKvChunkBytes = kTile * 128;       // 64 rows x 64 bf16
constexpr int kStageBytes = kChunks * kKvChunkBytes;
constexpr int kQChunkBytes = kHeads * 128;       // 128 rows x 64 bf16
constexpr int kPBytes = kHeads * 128;            // 128 heads x 64 tokens bf16 (one term)

constexpr int kOffKv = 0;
constexpr int kCodesPage = kTile * kDk;          // 8-bit cache: one page of E4M3 codes (36 KB)
// P of a tile (hi, then lo: 2 x 16 KB) lives in its own stage, in the four boxes
// of the other CTA's value dims (dims 256 (1-r) .. 256 (1-r) + 255), which this
// CTA reads only in the score MMA: one P buffer per stage, so writing P never
// waits for the previous tile's P.V.
// The 8-bit cache (F8) copies pages of E4M3 codes instead (36 KB, one bulk
// copy each, no multicast) into a one-page codes stage, and each page is
// widened, exactly, into fp16 boxes laid out like the bf16 ones: the five
// boxes only the score reads (the other CTA's value dims, by the softmax
// warps, and dims 512-575, by the producer warp) into one shared region,
// this CTA's four value boxes (softmax warps) into one of two value slots by
// page parity. P has a buffer of its own. So page g + 1
// can be widened as soon as page g's scores are read -- its score then runs
// while page g's softmax does -- the value slot it needs having been freed by
// the P.V of page g - 1.
constexpr int kNumBars = 22;
template <bool F8>
struct MlaLayout {
  static constexpr int kRing = F8 ? 1 : kStages;                 // copy stages
  static constexpr int kStage = F8 ? kCodesPage : kStageBytes;  // one copy stage
  static constexpr int kOffSh = kOffKv + kRing * kStage;          // F8: the score-only boxes (5)
  static constexpr int kOffV = kOffSh + (F8 ? 5 * kKvChunkBytes : 0);  // F8: own value boxes, 2 x 4
  static constexpr int kOffP = kOffV + (F8 ? 8 * kKvChunkBytes : 0);   // F8: P (hi, lo)
  static constexpr int kOffQ = kOffP + (F8 ? 2 * kPBytes : 0);
  static constexpr int kOffBar = kOffQ + kQSmemChunks * kQChunkBytes;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM slot, abort flag, residual votes (per stage)
  static constexpr int kOffLx = kOffMisc + 128;            // row-sum halves exchanged at the end of an item
  static constexpr int kOffMw = kOffLx + 2 * kHeads * 4;   // one-call path: merge weights [8 warps][16 heads][4]
  static constexpr int kSmemBytes = kOffMw + kSoftmaxWarps * 16 * kMlaMergeInKernel * 4 + 1024;  // + base alignment
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kOffSh % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 && kOffQ % 1024 == 0, "swizzle atoms");
};

// barrier slots
// BP_EMPTY + s: the P.V of the stage's latest tile finished (one per stage: the
// softmax waits on it only now and then, and a stage's barrier can never run
// more than one phase ahead of such a wait -- the tile after next in the same
// stage needs this tile's P.V to have finished before its page may land).
constexpr int BQ_FULL = 0, BQ_EMPTY = 1, BS_FULL = 2, BS_EMPTY = 3, BP_EMPTY = 4, BDRAIN = 6,
              BKV_FULL = 7, BKV_EMPTY = 7 + kStages, BXCH = 7 + 2 * kStages,  // BXCH: one per lane quadrant
              BDRAIN2 = BXCH + 4, BP_FULL = 16,  // BP_FULL + stage: the tile's P is in its stage
              BQT = BP_FULL + kStages,           // the copy of the query tail landed
              BF_FULL = BQT + 1,                 // F8: the page's widened boxes are in place
              BPC = BQT + 2,                     // one-call path: every softmax thread's piece rows are out
              BGO = BQT + 3;                     // one-call path: the piece is counted (merge or not)
static_assert(BDRAIN2 + 1 <= BP_FULL && BGO + 1 <= kNumBars, "barrier slots");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;       // 256 columns: O_r, fp32
constexpr uint32_t kColS = 256;     // 64 columns: S, fp32
constexpr uint32_t kColQ = 320;     // 192 columns: query dims 0-383, bf16 pairs

// Pages pulled into L2 ahead of the ring by CTA 0 of the pair (0: none); the
// ring's copies then find their page in L2 instead of waiting for HBM.
#ifndef DCP_MLA_PREFETCH_PAGES
#define DCP_MLA_PREFETCH_PAGES 4
#endif
constexpr int kPrefetch = DCP_MLA_PREFETCH_PAGES;
static_assert(kPrefetch >= 0 && kPrefetch <= 32, "prefetch distance within the table window");

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;       // log2 units
constexpr float kLoFraction = 1.0f / 32.0f;      // tile share of the row sum above which P_lo . V is issued

struct MlaParams {
  CUtensorMap tm_q;
  CUtensorMap tm_kv[kMaxShards];
  CUtensorMap tm_kv4[kMaxShards];  // token-split kernel: four 64-column boxes of a half page in one copy
  ShardSet sh;
  const __nv_bfloat16* q;
  const char* ws;
  WsLayout L;
  float* o_parts;
  float* lses;
  float* o;        // one-call path: merged rows [B][128][512] (NULL otherwise)
  float* lse_out;  // one-call path: merged LSEs (may be NULL)
  int32_t* err;
  int B;     // query rows: sequences x qlen
  int qlen;  // query tokens per sequence (block-table row = query row / qlen)
  float sl2;      // scale * log2(e) (x k_scale for the 8-bit cache)
  float v_scale;  // 8-bit cache: a value is v_scale * decode(code); 1 otherwise
};

// Shared geometry of one work item, derived identically by every role.
struct ItemGeom {
  int u, shard, b, t0, t1, out_row, lo, hi, start;
};
__device__ __forceinline__ ItemGeom item_geom(const MlaParams& p, int k) {
  const ItemRec it = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k];
  const LaneRec ln = reinterpret_cast<const LaneRec*>(p.ws + p.L.lanes_off)[it.lane];
  ItemGeom g;
  g.u = it.lane;
  g.shard = it.lane / p.B;
  g.b = it.lane - g.shard * p.B;
  g.t0 = it.t0;
  g.t1 = it.t1;
  g.out_row = it.out_row;
  g.lo = ln.lo;
  g.hi = ln.hi;
  g.start = ln.start;
  return g;
}
// Item k has the query rows of item k - 1 (the same row group, next shard:
// the plan lays a row group's shard lanes next to each other), so the query
// already in place serves it.
__device__ __forceinline__ bool same_rows(const MlaParams& p, int k, int k_begin) {
  if (k <= k_begin) return false;
  const ItemRec* items = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off);
  return items[k].lane % p.B == items[k - 1].lane % p.B;
}
// One-call path: item k also carries on the online softmax of item k - 1
// instead of starting afresh.
__device__ __forceinline__ bool continues(const MlaParams& p, int k, int k_begin) {
  return p.o != nullptr && same_rows(p, k, k_begin);
}

// One-call path: the CTA that completed the count of a row group cut into at
// most kMlaMergeInKernel pieces merges the pieces' value dims [256 rank,
// 256 rank + 256) into o (the LSE reweighting: M = max LSE_i, w_i =
// e^(LSE_i - M), O = sum w_i O_i / sum w_i, LSE = M + ln sum w_i). The 256
// softmax threads: warp w takes heads 16 w .. 16 w + 15, lane l columns
// 4l .. 4l + 3 and 128 + 4l ..; loads bypass L1 (the pieces were written by
// other SMs). Its cost is dependent L2 round trips: the weights of the
// warp's 16 heads come from one round of loads (lane k: piece k's LSEs) and
// wait in shared memory, and the pieces of two or four heads are loaded
// together.
template <int HB, int KB>  // heads per batch, pieces per batch (>= the group's pieces)
__device__ __forceinline__ void merge_rows(const MlaParams& p, const float* tmp_o, int rg, int tmp_begin, int n,
                                           uint32_t rank, int h0, int lane, const float* wt) {
#pragma unroll 1
  for (int i0 = 0; i0 < 16; i0 += HB) {
    float4 v0[HB][KB], v1[HB][KB];
#pragma unroll
    for (int hb = 0; hb < HB; ++hb)
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        v0[hb][k] = v1[hb][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < n) {
          const float4* src = reinterpret_cast<const float4*>(
              tmp_o + ((size_t)(tmp_begin + k) * kHeads + h0 + i0 + hb) * kDv + 256 * rank);
          v0[hb][k] = __ldcg(src + lane);
          v1[hb][k] = __ldcg(src + 32 + lane);
        }
      }
#pragma unroll
    for (int hb = 0; hb < HB; ++hb) {
      float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        const float w = k < n ? wt[(i0 + hb) * kMlaMergeInKernel + k] : 0.f;
        a0 = make_float4(fmaf(w, v0[hb][k].x, a0.x), fmaf(w, v0[hb][k].y, a0.y), fmaf(w, v0[hb][k].z, a0.z),
                         fmaf(w, v0[hb][k].w, a0.w));
        a1 = make_float4(fmaf(w, v1[hb][k].x, a1.x), fmaf(w, v1[hb][k].y, a1.y), fmaf(w, v1[hb][k].z, a1.z),
                         fmaf(w, v1[hb][k].w, a1.w));
      }
      float4* dst = reinterpret_cast<float4*>(p.o + ((size_t)rg * kHeads + h0 + i0 + hb) * kDv + 256 * rank);
      dst[lane] = a0;
      dst[32 + lane] = a1;
    }
  }
}

__device__ __forceinline__ void merge_pieces(const MlaParams& p, int rg, int tmp_begin, int n, uint32_t rank, int warp,
                                          int lane, float* mw) {
  const float* tmp_o = reinterpret_cast<const float*>(p.ws + p.L.tmp_o_off);
  const float* tmp_lse = reinterpret_cast<const float*>(p.ws + p.L.tmp_lse_off);
  const int h0 = 16 * warp;
  float lv[16];
  if (lane < n) {
    const float4* src = reinterpret_cast<const float4*>(tmp_lse + (size_t)(tmp_begin + lane) * kHeads + h0);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 v = __ldcg(src + c);
      lv[4 * c] = v.x;
      lv[4 * c + 1] = v.y;
      lv[4 * c + 2] = v.z;
      lv[4 * c + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) lv[i] = -INFINITY;
  }
  float* wt = mw + warp * 16 * kMlaMergeInKernel;  // [head][piece]: normalised weights
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float M = lv[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = (M == -INFINITY || lv[i] == -INFINITY) ? 0.f : expf(lv[i] - M);
    float ws = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    if (lane < kMlaMergeInKernel) wt[i * kMlaMergeInKernel + lane] = ws > 0.f ? w / ws : 0.f;
    if (rank == 0 && lane == 0 && p.lse_out)
      p.lse_out[(size_t)rg * kHeads + h0 + i] = ws > 0.f ? M + logf(ws) : -INFINITY;
  }
  __syncwarp();
  if (n <= 2)
    merge_rows<4, 2>(p, tmp_o, rg, tmp_begin, n, rank, h0, lane, wt);
  else
    merge_rows<2, kMlaMergeInKernel>(p, tmp_o, rg, tmp_begin, n, rank, h0, lane, wt);
  __syncwarp();
}

// Physical block of tile t of the item, or -1 if the table entry is unusable.
__device__ __forceinline__ int tile_block(const MlaParams& p, const ItemGeom& g, int t) {
  const int lb = (g.lo - g.start) / kTile + t;
  if (lb >= p.sh.max_blocks[g.shard]) return -1;
  const int phys = p.sh.table[g.shard][(size_t)(g.b / p.qlen) * p.sh.max_blocks[g.shard] + lb];
  return (phys < 0 || phys >= p.sh.nblk[g.shard]) ? -1 : phys;
}

// hi = fp16(x), lo = fp16(x - hi) for a pair (x0 in the low half): P of the
// 8-bit cache's fp16 MMAs carries ~22 mantissa bits; x >= 0, below 2^15.
__device__ __forceinline__ void split_p_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// bf16 pair -> fp16 pair (round to nearest; the query of the 8-bit cache's
// fp16 MMAs, |q| below 65504)
__device__ __forceinline__ uint32_t bf16x2_as_f16x2(uint32_t v) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  const __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 lds128_u32(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
// four E4M3 codes (low byte first) -> two fp16 pairs, exactly: codes 0, 1 ->
// lo, codes 2, 3 -> hi
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

template <bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_partial_kernel(const __grid_constant__ MlaParams p) {
  using Lay = MlaLayout<F8>;
  constexpr int kOffQ = Lay::kOffQ, kOffBar = Lay::kOffBar, kOffMisc = Lay::kOffMisc, kOffLx = Lay::kOffLx;
  constexpr int kStage = Lay::kStage, kRing = Lay::kRing;
  constexpr int kOffSh = Lay::kOffSh, kOffV = Lay::kOffV, kOffP = Lay::kOffP;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = saddr(smem);
  const uint32_t rank = cluster_rank();
  const int cluster = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* lo_flags = reinterpret_cast<volatile int*>(smem + kOffMisc + 16);  // [stage][softmax warp]
  // F8: each page's physical block as the producer read it (ring of 4,
  // written before the page's copy barrier is arrived on), so that the
  // softmax warps make no block-table load of their own
  volatile int* phys_ring = reinterpret_cast<volatile int*>(smem + kOffMisc + 80);

  if (threadIdx.x == 0) {
    bar_init(bar(BQ_FULL), kSoftmaxThreads);  // every softmax thread's share of Q[:, 0:384] in TMEM
    bar_init(bar(BQT), 1);                    // the producer's copy of Q[:, 384:576]
    bar_init(bar(BQ_EMPTY), 1);
    bar_init(bar(BS_FULL), 1);
    bar_init(bar(BS_EMPTY), kSoftmaxThreads);
    for (int s = 0; s < kStages; ++s) bar_init(bar(BP_FULL + s), kSoftmaxThreads);
    for (int s = 0; s < kStages; ++s) bar_init(bar(BP_EMPTY + s), 1);
    bar_init(bar(BDRAIN), 1);
    bar_init(bar(BDRAIN2), 1);
    for (int s = 0; s < kRing; ++s) {
      bar_init(bar(BKV_FULL + s), 1);
      // bf16: the P.V of both CTAs (the page lands in both); F8: the widening of the codes
      bar_init(bar(BKV_EMPTY + s), F8 ? kSoftmaxThreads + 1 : 2);  // F8: + the producer's rope box
    }
    for (int q4 = 0; q4 < 4; ++q4) bar_init(bar(BXCH + q4), 64);  // the two warps of a lane quadrant
    bar_init(bar(BF_FULL), kSoftmaxThreads + 1);  // the softmax threads and the producer (rope box)
    bar_init(bar(BPC), kSoftmaxThreads);
    bar_init(bar(BGO), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(saddr(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either copies into the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int* cta_begin = reinterpret_cast<const int*>(p.ws + p.L.cta_off);
  const int k_begin = cta_begin[cluster], k_end = cta_begin[cluster + 1];

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // The whole warp reads block-table entries 32 tiles at a time (lane i
    // holds tile base + i); lane 0 issues the copies.
    uint32_t fills = 0;  // K/V tiles issued (global across items)
    int q_done = 0;      // query tails copied
    bool stop = false;
    for (int k = k_begin; k < k_end && !stop; ++k) {
      const ItemGeom g = item_geom(p, k);
      const int nt = g.t1 - g.t0;
      const bool same_q = same_rows(p, k, k_begin);  // the query in place serves this item too
      // the next row group's query into L2 while this item runs (its load is
      // a few dependent round trips at the next item boundary otherwise)
      if (lane == 0 && rank == 0 && k + 1 < k_end && !same_rows(p, k + 1, k_begin)) {
        const int nb = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k + 1].lane % p.B;
        l2_prefetch(p.q + (size_t)nb * kHeads * kDk, kHeads * kDk * 2);
      }
      int cur = lane < nt ? tile_block(p, g, g.t0 + lane) : -1;
      int nxt = 32 + lane < nt ? tile_block(p, g, g.t0 + 32 + lane) : -1;
      bool ok = true;
      if (lane == 0) {
        if (F8 || same_q) {
          // (F8: the softmax warps write the fp16 query tail themselves)
        } else if (q_done > 0 && !wait_bar(bar(BQ_EMPTY), (q_done - 1) & 1, abort_flag, p.err, false)) {
          ok = false;
        } else {
          bar_arrive_tx(bar(BQT), kQSmemChunks * kQChunkBytes);
          for (int c = 0; c < kQSmemChunks; ++c)
            tma_load(sbase + kOffQ + c * kQChunkBytes, &p.tm_q, 384 + 64 * c, g.b * kHeads, bar(BQT));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) { stop = true; break; }
      if (!F8 && !same_q) ++q_done;
      for (int j = 0; j < nt; ++j) {
        if ((j & 31) == 0 && j > 0) {
          cur = nxt;
          nxt = j + 32 + lane < nt ? tile_block(p, g, g.t0 + j + 32 + lane) : -1;
        }
        const int phys = __shfl_sync(0xffffffffu, cur, j & 31);
        int phys_pf = -1;
        if (kPrefetch > 0) {  // tile j + kPrefetch sits in this window of 32 table entries or the next
          const int jp = j + kPrefetch;
          const int a = __shfl_sync(0xffffffffu, cur, jp & 31), b2 = __shfl_sync(0xffffffffu, nxt, jp & 31);
          phys_pf = jp < nt ? ((jp >> 5) == (j >> 5) ? a : b2) : -1;
        }
        if (lane == 0) {
          const uint32_t s = fills % kRing, use = fills / kRing;
          if (use > 0 && !wait_bar(bar(BKV_EMPTY + s), (use - 1) & 1u, abort_flag, p.err, false)) {
            ok = false;
          } else {
            if (phys < 0 && rank == 0) raise_flag(p.err, DCP_DEVERR_BLOCK_RANGE);
            if constexpr (F8) {
              // one bulk copy of the page's codes (an unusable table entry
              // copies nothing: the widening writes zeros for it)
              phys_ring[fills & 3u] = phys;
              if (phys < 0) {
                bar_arrive(bar(BKV_FULL + s));
              } else {
                bar_arrive_tx(bar(BKV_FULL + s), kCodesPage);
                bulk_load(sbase + kOffKv + s * kStage,
                          static_cast<const unsigned char*>(p.sh.k[g.shard]) + (size_t)phys * kCodesPage, kCodesPage,
                          bar(BKV_FULL + s));
              }
            } else {
              const int row = phys < 0 ? -kTile : phys * kTile;  // out of range: the copy reads zeros
              // the pair copies each page once: each CTA fetches alternate boxes
              // into both CTAs (one L2 read per box); every CTA's barrier
              // expects the whole page
              bar_arrive_tx(bar(BKV_FULL + s), kChunks * kKvChunkBytes);
              for (int c = (int)rank; c < kChunks; c += 2)
                tma_load_mc(sbase + kOffKv + s * kStageBytes + c * kKvChunkBytes, &p.tm_kv[g.shard], 64 * c, row,
                            bar(BKV_FULL + s), 0x3);
            }
            if (kPrefetch > 0 && rank == 0 && phys_pf >= 0)
              l2_prefetch(static_cast<const char*>(p.sh.k[g.shard]) + (size_t)phys_pf * kStage, kStage);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) { stop = true; break; }
        if constexpr (F8) {
          // F8: the producer widens box 8 (dims 512-575) of this page into
          // the score-only region itself, once the codes have landed and the
          // previous page's score has finished with that region, so that the
          // softmax warps widen eight boxes instead of nine (same layout and
          // zero rows as theirs: 64 rows x four 16-code pieces, 8 per lane)
          const uint32_t G = fills;
          const int n_rows = phys < 0 ? 0 : min(kTile, g.hi - (g.lo + kTile * (g.t0 + j)));
          if (!wait_warp(bar(BKV_FULL), G & 1u, abort_flag, p.err, false) ||
              (G > 0 && !wait_warp(bar(BS_FULL), (G - 1) & 1u, abort_flag, p.err, false))) {
            stop = true;
            break;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int w = lane + 32 * i, r = w >> 2, q4 = w & 3;
            const uint32_t sw = (uint32_t)(r & 7), ch = 2u * (uint32_t)q4;
            const uint32_t dst = sbase + kOffSh + 4 * kKvChunkBytes + r * 128;
            uint32_t wv[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (r < n_rows) {
              const uint4 c = lds128_u32(sbase + kOffKv + r * kDk + 512 + 16 * q4);
              e4m3x4_to_f16x4(c.x, wv[0], wv[1]);
              e4m3x4_to_f16x4(c.y, wv[2], wv[3]);
              e4m3x4_to_f16x4(c.z, wv[4], wv[5]);
              e4m3x4_to_f16x4(c.w, wv[6], wv[7]);
            }
            st_shared_v4(dst + ((ch ^ sw) << 4), wv[0], wv[1], wv[2], wv[3]);
            st_shared_v4(dst + (((ch + 1) ^ sw) << 4), wv[4], wv[5], wv[6], wv[7]);
          }
          asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            bar_arrive(bar(BF_FULL));
            bar_arrive(bar(BKV_EMPTY));  // done with the codes
          }
        }
        ++fills;
      }
    }
    if (lane == 0 && *abort_flag) {  // copies in flight must land before the CTA may exit
      if (!F8 && q_done > 0) drain_bar(bar(BQT), (q_done - 1) & 1u);
      // (the other CTA's copies into this one land on the same barriers; it
      // can be at most one page ahead, which may never complete here: the
      // poll bound ends that wait)
      const uint32_t f0 = fills > (uint32_t)kRing ? fills - kRing : 0;
      for (uint32_t f = f0; f < fills + 1; ++f) drain_bar(bar(BKV_FULL + f % kRing), (f / kRing) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ score MMA issuer
    // The whole warp runs the loop (uniform control flow); one elected lane
    // issues. The P.V products come from a warp of their own (below), so a
    // ready P.V enters the tensor pipe while a score is being issued instead
    // of waiting for all its 36 MMAs.
    {
      const uint32_t id_s = idesc(128, 64, 0, F8);
      const uint64_t kdesc0 = sdesc(sbase + (F8 ? kOffSh : kOffKv), 0);
      const uint64_t qdesc0 = sdesc(sbase + kOffQ, 0);
      // F8: this CTA's value boxes of even / odd pages
      const uint64_t vdesc_e = sdesc(sbase + kOffV, 0), vdesc_o = sdesc(sbase + kOffV + 4 * kKvChunkBytes, 0);
      auto n_tiles = [&](int k) {
        const ItemRec it = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k];
        return it.t1 - it.t0;
      };
      int ks = k_begin, js = 0, nts = ks < k_end ? n_tiles(ks) : 0;  // next score tile
      uint32_t g_s = 0, q_loads = 0;
      bool q_ready = false;
      uint32_t idle = 0;
      while (ks < k_end) {
        bool progressed = false;
        if (!q_ready && bar_test_warp(bar(BQ_FULL), q_loads & 1u) && (F8 || bar_test_warp(bar(BQT), q_loads & 1u))) {
          q_ready = true;
          tc_fence_after();
        }
        const uint32_t s = g_s % kStages;
        const bool page_in = F8 ? bar_test_warp(bar(BF_FULL), g_s & 1u)  // the widened page
                                : bar_test_warp(bar(BKV_FULL + s), (g_s / kStages) & 1u);
        if (q_ready && page_in && (g_s == 0 || bar_test_warp(bar(BS_EMPTY), (g_s - 1) & 1u))) {
          tc_fence_after();
          // descriptors advance by (byte offset >> 4) in their address field
          const uint64_t kd = kdesc0 + (F8 ? 0ull : (uint64_t)((s * kStageBytes) >> 4));
          const uint64_t kv = (g_s & 1u) ? vdesc_o : vdesc_e;
#pragma unroll
          for (int kk = 0; kk < kKSteps; ++kk) {
            const int box = kk >> 2;
            uint64_t bdesc;
            if constexpr (F8) {
              // this CTA's value boxes in the page's value slot; the other
              // CTA's value boxes and box 8 (slot 4) in the shared region
              const bool own = (box >> 2) == (int)rank;
              const int slot = box == 8 ? 4 : (box & 3);
              bdesc = (own ? kv : kd) + (uint64_t)((slot * kKvChunkBytes + 32 * (kk & 3)) >> 4);
            } else {
              bdesc = kd + (uint64_t)(((box * kKvChunkBytes) + 32 * (kk & 3)) >> 4);
            }
            if (kk < kKStepsTmem) {
              mma_ts(tmem + kColS, tmem + kColQ + 8 * kk, bdesc, id_s, kk > 0);
            } else {
              const int qk = kk - kKStepsTmem;
              mma_ss(tmem + kColS, qdesc0 + (uint64_t)((((qk >> 2) * kQChunkBytes) + 32 * (qk & 3)) >> 4), bdesc,
                  id_s, 1);
            }
          }
          mma_commit(bar(BS_FULL));
          if (++js == nts) {  // last score tile of the item
            if (!(ks + 1 < k_end && same_rows(p, ks + 1, k_begin))) {  // its queries may be replaced
              mma_commit(bar(BQ_EMPTY));
              ++q_loads;
              q_ready = false;
            }
            ++ks;
            js = 0;
            nts = ks < k_end ? n_tiles(ks) : 0;
          }
          ++g_s;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle >= kSpinLimit) {
          *abort_flag = 1;
          raise_flag(p.err, DCP_DEVERR_TIMEOUT);
          break;
        } else if ((idle & 63u) == 0 && __any_sync(0xffffffffu, *abort_flag != 0)) {
          break;
        }
      }
      mma_commit(bar(BDRAIN));  // this warp's MMAs complete before TMEM may be freed
      drain_bar(bar(BDRAIN), 0);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P.V MMA issuer
    // Waits for each tile's P in order. BP_FULL + s's phase for tile g (stage
    // s = g % kStages) completes only after the stage was refilled, i.e. after
    // the P.V of tile g - kStages, so this warp is never more than one phase
    // behind on either barrier and its parity waits are unambiguous.
    {
      const uint32_t id_pv = idesc(128, 256, 1, F8);
      // bf16: P in the stage's dead boxes, V in the stage; F8: P in its own
      // buffer, V in the page parity's value slot
      const uint64_t pdesc0 = sdesc(F8 ? sbase + kOffP : sbase + kOffKv + 4 * (1 - rank) * kKvChunkBytes, 0);
      const uint64_t vdesc0 = sdesc(F8 ? sbase + kOffV : sbase + kOffKv + 4 * rank * kKvChunkBytes, kKvChunkBytes);
      auto n_tiles = [&](int k) {
        const ItemRec it = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k];
        return it.t1 - it.t0;
      };
      int kp = k_begin, jp = 0, ntp = kp < k_end ? n_tiles(kp) : 0;  // next P.V tile
      bool acc_in = false;  // the item's first P.V adds to O (it carries on the previous item)
      uint32_t g_p = 0;
      uint32_t idle = 0;
      while (kp < k_end) {
        const uint32_t s = g_p % kStages;
        if (bar_test_warp(bar(BP_FULL + s), (g_p / kStages) & 1u)) {
          tc_fence_after();
          const uint64_t soff = (uint64_t)((s * kStageBytes) >> 4);
          const uint64_t vd = vdesc0 + (F8 ? (uint64_t)(((g_p & 1u) * 4 * kKvChunkBytes) >> 4) : soff);  // V dims of this CTA
          const uint64_t pd = pdesc0 + (F8 ? 0ull : soff);  // P of this tile
          int any_lo = 0;
#pragma unroll
          for (int w = 0; w < kSoftmaxWarps; ++w) any_lo |= lo_flags[kSoftmaxWarps * s + w];
          const int terms = any_lo ? 2 : 1;
#pragma unroll
          for (int term = 0; term < 2; ++term) {
            if (term >= terms) break;
#pragma unroll
            for (int kt = 0; kt < kTile / 16; ++kt)
              mma_ss(tmem + kColO, pd + (uint64_t)((term * kPBytes + 32 * kt) >> 4),
                  vd + (uint64_t)((2048 * kt) >> 4), id_pv, (jp == 0 && !acc_in && term == 0 && kt == 0) ? 0 : 1);
          }
          if (!F8) mma_commit_mc(bar(BKV_EMPTY + s), 0x3);  // the stage is free in both CTAs once both P.V finished
          // (F8: the value slot and P may be overwritten)
          mma_commit(bar(BP_EMPTY + s));  // also tells softmax that this P.V finished
          if (++jp == ntp) {
            ++kp;
            jp = 0;
            ntp = kp < k_end ? n_tiles(kp) : 0;
            acc_in = kp < k_end && continues(p, kp, k_begin);
          }
          ++g_p;
          idle = 0;
        } else if (++idle >= kSpinLimit) {
          *abort_flag = 1;
          raise_flag(p.err, DCP_DEVERR_TIMEOUT);
          break;
        } else if ((idle & 63u) == 0 && __any_sync(0xffffffffu, *abort_flag != 0)) {
          break;
        }
      }
      mma_commit(bar(BDRAIN2));  // this warp's MMAs complete before TMEM may be freed
      drain_bar(bar(BDRAIN2), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // Warp w owns TMEM lane quadrant qd = w % 4 (query heads 32 qd .. 32 qd + 31,
    // one per lane) and half e = w / 4: the tile's tokens 32 e .. 32 e + 31 for
    // the exponentials and P, and this CTA's value dims 128 e .. 128 e + 127 of
    // O. Both warps of a quadrant read all 64 scores of their rows and take
    // the same maximum, so they hold the same running max without talking to
    // each other; each keeps the row sum of its own tokens, and the two sums
    // are added once per item, through shared memory, for the epilogue.
    const int qd = warp & 3, e = warp >> 2;
    const int h = 32 * qd + lane;  // query head = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
    const int vlo = 4 * (int)rank;  // first V box of this CTA
    const bool pos_scale = p.sl2 >= 0.f;
    float* lx = reinterpret_cast<float*>(smem + kOffLx);  // [2][kHeads] row-sum halves
    uint32_t gt = 0;
    int n_q = 0, n_epi = 0;  // query loads, epilogues
    uint32_t n_pc = 0;       // pieces counted (one-call path)
    float m_run = -INFINITY, l_half = 0.f;
    volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 96);
    // F8: widen page G's codes (in the codes stage) to fp16, exactly (E4M3 is
    // a subset of fp16): part 0 the score-only boxes into the shared region,
    // part 1 this CTA's value boxes into the value slot of G's parity. Rows
    // past the range (or of an unusable table entry) become zeros, so that no
    // value can carry NaN bits. Four threads per row (thread = row 4r + q),
    // 16 codes per load: codes 16 (q + 4i) .. + 15 -> box i, 16-byte chunks
    // 2q, 2q + 1.
    auto widen = [&](uint32_t G, int n_rows, int part) {
      const int r = threadIdx.x >> 2, q4 = threadIdx.x & 3;
      const uint32_t src = sbase + kOffKv + r * kDk + 16 * q4;
      const uint32_t sw = (uint32_t)(r & 7), ch = 2u * (uint32_t)q4;
      const uint32_t c0 = (ch ^ sw) << 4, c1 = ((ch + 1) ^ sw) << 4;
      const bool live = r < n_rows;
      // part 0: the other CTA's value boxes 4 (1 - rank) + i (i < 4) into
      // slots i of the shared region (box 8, slot 4, is the producer's);
      // part 1: this CTA's value boxes 4 rank + i into the value slot of
      // G's parity
      const uint32_t dst0 = (part == 0 ? sbase + kOffSh : sbase + kOffV + (G & 1u) * 4 * kKvChunkBytes) + r * 128;
      const int box0 = part == 0 ? 4 * (1 - (int)rank) : 4 * (int)rank;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int box = box0 + i;
        const uint32_t dst = dst0 + i * kKvChunkBytes;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (live) {
          const uint4 c = lds128_u32(src + 64 * box);
          e4m3x4_to_f16x4(c.x, w[0], w[1]);
          e4m3x4_to_f16x4(c.y, w[2], w[3]);
          e4m3x4_to_f16x4(c.z, w[4], w[5]);
          e4m3x4_to_f16x4(c.w, w[6], w[7]);
        }
        st_shared_v4(dst + c0, w[0], w[1], w[2], w[3]);
        st_shared_v4(dst + c1, w[4], w[5], w[6], w[7]);
      }
    };
    bool ok = true;
    for (int k = k_begin; k < k_end && ok; ++k) {
      const ItemGeom g = item_geom(p, k);
      const int nt = g.t1 - g.t0;
      if (!same_rows(p, k, k_begin)) {  // a new query row group: its query
        // query dims 192 e .. 192 e + 191 of this item into TMEM (after the previous item's score MMAs)
        if (n_q > 0 && !wait_warp(bar(BQ_EMPTY), (n_q - 1) & 1, abort_flag, p.err, false)) break;
        tc_fence_after();
        {
          const uint4* qr = reinterpret_cast<const uint4*>(p.q + ((size_t)g.b * kHeads + h) * kDk + 192 * e);
          uint32_t qv[16];
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < 6; ++c) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 v = qr[4 * c + i];
              qv[4 * i] = F8 ? bf16x2_as_f16x2(v.x) : v.x;
              qv[4 * i + 1] = F8 ? bf16x2_as_f16x2(v.y) : v.y;
              qv[4 * i + 2] = F8 ? bf16x2_as_f16x2(v.z) : v.z;
              qv[4 * i + 3] = F8 ? bf16x2_as_f16x2(v.w) : v.w;
            }
            tmem_st16(tmem + lane_off + kColQ + 96 * e + 16 * c, qv);
          }
          tmem_wait_st();
          if constexpr (F8) {
            // query dims 384 + 96 e .. + 95 in fp16 into the shared-memory tail
            // (128-byte swizzled rows of 64 dims, as the copy would lay them out)
            const uint4* qt = reinterpret_cast<const uint4*>(p.q + ((size_t)g.b * kHeads + h) * kDk + 384 + 96 * e);
#pragma unroll 4
            for (int c = 0; c < 12; ++c) {
              const uint4 v = qt[c];
              const int d = 96 * e + 8 * c;  // dim - 384
              const uint32_t a = sbase + kOffQ + (d >> 6) * kQChunkBytes + h * 128 +
                                 (((uint32_t)((d & 63) >> 3) ^ (uint32_t)(h & 7)) << 4);
              st_shared_v4(a, bf16x2_as_f16x2(v.x), bf16x2_as_f16x2(v.y), bf16x2_as_f16x2(v.z), bf16x2_as_f16x2(v.w));
            }
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
          }
        }
        tc_fence_before();
        bar_arrive(bar(BQ_FULL));
        ++n_q;
      }
      if (!continues(p, k, k_begin)) {  // a fresh softmax
        m_run = -INFINITY;
        l_half = 0.f;
      }
      for (int j = 0; j < nt; ++j) {
        const uint32_t gi = gt + j, s = gi % kStages;
        const int t = g.t0 + j;
        int phys;  // bf16: its latency hides behind the score wait; F8: from the ring
        if constexpr (F8) {
          if (gi == 0) {  // 0. the run's first page is widened before its score
            if (!wait_warp(bar(BKV_FULL), 0u, abort_flag, p.err, false)) { ok = false; break; }
            phys = phys_ring[0];
            const int n_rows = phys < 0 ? 0 : min(kTile, g.hi - (g.lo + kTile * t));
            widen(0u, n_rows, 0);
            widen(0u, n_rows, 1);
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            bar_arrive(bar(BF_FULL));
            bar_arrive(bar(BKV_EMPTY));  // the codes' stage may be refilled
          } else {
            phys = phys_ring[gi & 3u];  // written before the page's copy barrier, which was waited for
          }
        } else {
          phys = tile_block(p, g, t);
        }
        // 1. scores of the tile: all 64 for the maximum, this warp's 32 for P
        if (!wait_warp(bar(BS_FULL), gi & 1u, abort_flag, p.err, false)) { ok = false; break; }
        tc_fence_after();
        // sv[0..31]: this warp's tokens 32 e .., sv[32..63]: the other half's
        uint32_t sv[64];
        __syncwarp();
        tmem_ld32(tmem + lane_off + kColS + 32 * e, sv);
        tmem_ld32(tmem + lane_off + kColS + 32 * (1 - e), sv + 32);
        tmem_wait_ld();
        tc_fence_before();
        bar_arrive(bar(BS_EMPTY));
        if constexpr (F8) {
          // 1b. widen the next page (this item's next tile, or the next
          // item's first) now, so that its score runs during this page's
          // softmax: the score-only boxes at once (this page's score has
          // finished with them), this CTA's value boxes once the P.V of the
          // page before this one has finished with their slot
          int tn = -1;
          ItemGeom gn = g;
          if (j + 1 < nt) {
            tn = t + 1;
          } else if (k + 1 < k_end) {
            gn = item_geom(p, k + 1);
            tn = gn.t0;
          }
          if (tn >= 0) {
            const uint32_t G = gi + 1;
            if (!wait_warp(bar(BKV_FULL), G & 1u, abort_flag, p.err, false)) { ok = false; break; }
            const int physn = phys_ring[G & 3u];
            const int n_rows = physn < 0 ? 0 : min(kTile, gn.hi - (gn.lo + kTile * tn));
            widen(G, n_rows, 0);
            if (G >= 2 && !wait_warp(bar(BP_EMPTY + (G & 1u)), ((G - 2) >> 1) & 1u, abort_flag, p.err, false)) {
              ok = false;
              break;
            }
            widen(G, n_rows, 1);
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            bar_arrive(bar(BF_FULL));
            bar_arrive(bar(BKV_EMPTY));  // the codes' stage may be refilled
          }
        }
        // 2. online softmax (log2 units). The maximum of scale * s is taken as
        // scale * max(s) (or * min(s) for a negative scale): one multiply.
        const int n_valid = phys < 0 ? 0 : min(kTile, g.hi - (g.lo + kTile * t));
        float raw_ext;
        if (n_valid == kTile) {  // common case: no masking; a tree of three-input extrema
          raw_ext = pos_scale ? ext_tree<64, true>(sv) : ext_tree<64, false>(sv);
        } else {
          raw_ext = pos_scale ? -INFINITY : INFINITY;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const float x = __uint_as_float(sv[i]);
            const int tok = i < 32 ? 32 * e + i : 32 * (1 - e) + (i - 32);
            if (tok < n_valid) raw_ext = pos_scale ? fmaxf(raw_ext, x) : fminf(raw_ext, x);
          }
        }
        // an empty tile leaves raw_ext infinite; its scaled max is -inf
        const float mx = n_valid > 0 ? raw_ext * p.sl2 : -INFINITY;
        float m_new = m_run, alpha = 1.f;
        bool rescale = false;
        if (m_run == -INFINITY) {
          m_new = mx;
        } else if (mx > m_run + kRescaleThreshold) {
          m_new = mx;
          alpha = exp2f(m_run - m_new);
          rescale = true;
        }
        const float ref = m_new == -INFINITY ? 0.f : m_new;
        float sc[32];
        float lsum;
        {
          // two scores scaled and shifted per instruction; the row sum in pairs
          const int t0 = 32 * e;
          const unsigned long long s2 = f2pack(p.sl2, p.sl2), r2 = f2pack(-ref, -ref);
          unsigned long long a0 = f2pack(0.f, 0.f), a1 = a0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), s2, r2), x0, x1);
            sc[2 * i] = (t0 + 2 * i < n_valid) ? ex2_ftz(x0) : 0.f;
            sc[2 * i + 1] = (t0 + 2 * i + 1 < n_valid) ? ex2_ftz(x1) : 0.f;
            if (i & 1)
              a1 = fadd2(a1, f2pack(sc[2 * i], sc[2 * i + 1]));
            else
              a0 = fadd2(a0, f2pack(sc[2 * i], sc[2 * i + 1]));
          }
          float y0, y1;
          f2unpack(fadd2(a0, a1), y0, y1);
          lsum = y0 + y1;
        }
        l_half = l_half * alpha + lsum;
        m_run = m_new;
        // The residual term matters only where this tile carries a noticeable
        // share of the row's weight (the first tiles of an item, or a tile
        // with a dominant token); elsewhere its P.V is skipped. Each warp
        // judges its own tokens against its own running sum (a share of a
        // part of the row bounds the share of the whole row). The residual
        // itself is stored for every row on every tile: the P.V covers all
        // 128 rows, so when any warp asks for it, every row must be current.
        const bool any_lo = __any_sync(0xffffffffu, lsum > kLoFraction * l_half);
        // 3. P into its stage (the score MMA that read those boxes has finished;
        // F8: into the P buffer, as fp16 terms, once the previous page's P.V
        // has finished with it -- mostly already waited for by the widening)
        if (F8 && gi >= 1 &&
            !wait_warp(bar(BP_EMPTY + (gi - 1) % kStages), ((gi - 1) / kStages) & 1u, abort_flag, p.err, false)) {
          ok = false;
          break;
        }
        {
          const uint32_t hrow =
              (F8 ? sbase + kOffP : sbase + kOffKv + s * kStageBytes + 4 * (1 - rank) * kKvChunkBytes) + h * 128;
          const uint32_t lrow = hrow + kPBytes;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t chunk = (uint32_t)(4 * e + c);
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              if constexpr (F8)
                split_p_f16(sc[8 * c + 2 * k2], sc[8 * c + 2 * k2 + 1], hi[k2], lo[k2]);
              else
                split_p_bf16(sc[8 * c + 2 * k2], sc[8 * c + 2 * k2 + 1], hi[k2], lo[k2]);
            }
            st_shared_v4(hrow + ((chunk ^ (uint32_t)(h & 7)) << 4), hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(lrow + ((chunk ^ (uint32_t)(h & 7)) << 4), lo[0], lo[1], lo[2], lo[3]);
          }
          if (lane == 0) lo_flags[kSoftmaxWarps * s + warp] = any_lo ? 1 : 0;
        }
        // 4. V rows past the end of a partial tile may hold anything: zero them
        // (F8: the widening already wrote zeros there)
        if (!F8 && n_valid < kTile) {
          const int rows = kTile - n_valid;
          const int tid = threadIdx.x;  // 0 .. kSoftmaxThreads-1
          for (int x = tid; x < rows * 4 * 8; x += kSoftmaxThreads) {
            const int r = n_valid + x / 32, c = vlo + ((x >> 3) & 3), piece = x & 7;
            st_shared_v4(sbase + kOffKv + s * kStageBytes + c * kKvChunkBytes + r * 128 + piece * 16, 0u, 0u, 0u, 0u);
          }
        }
        // 5. lazy rescale of this warp's half of O (warp-wide: TMEM access is per
        // warp; rows that did not grow multiply by 1), once the previous
        // tile's P.V has finished accumulating into it.
        if (__any_sync(0xffffffffu, rescale)) {
          if (gi >= 1 && !wait_warp(bar(BP_EMPTY + (gi - 1) % kStages), ((gi - 1) / kStages) & 1u, abort_flag, p.err,
                                    false)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t ov[32];
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            const uint32_t col = kColO + 128 * e + 32 * c;
            tmem_ld32(tmem + lane_off + col, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tmem + lane_off + col, ov);
          }
          tmem_wait_st();
        }
        // 6. publish P to the MMA issuer
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        tc_fence_before();
        bar_arrive(bar(BP_FULL + s));
      }
      if (!ok) break;
      if (k + 1 < k_end && continues(p, k + 1, k_begin)) {  // the next shard carries on this softmax
        gt += nt;
        continue;
      }
      // epilogue: the row sum of the two halves, then wait for the last P.V
      // and write this warp's dims of O_r / l and the LSE
      lx[e * kHeads + h] = l_half;
      bar_arrive(bar(BXCH + qd));  // release: the partner reads lx after its wait
      if (!wait_warp(bar(BXCH + qd), (uint32_t)n_epi & 1u, abort_flag, p.err, false)) break;
      const float l_run = l_half + lx[(1 - e) * kHeads + h];
      const uint32_t glast = gt + nt - 1;
      // (P.V products finish in issue order: the last one implies the others)
      if (!wait_warp(bar(BP_EMPTY + glast % kStages), (glast / kStages) & 1u, abort_flag, p.err, false)) break;
      tc_fence_after();
      const float inv = l_run > 0.f ? p.v_scale / l_run : 0.f;
      float* out;
      float* out_lse;
      GroupRec gr;
      bool piece = false;  // one-call path, row group cut by a CTA run boundary
      if (p.o) {
        gr = reinterpret_cast<const GroupRec*>(p.ws + p.L.grp_off)[g.b];
        piece = gr.pieces > 1;
        if (piece) {
          const size_t row = (size_t)(gr.tmp_begin + cluster - gr.first_cta);
          out = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_o_off) + (row * kHeads + h) * kDv;
          out_lse = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_lse_off) + row * kHeads + h;
        } else {
          out = p.o + ((size_t)g.b * kHeads + h) * kDv;
          out_lse = p.lse_out ? p.lse_out + (size_t)g.b * kHeads + h : nullptr;
        }
      } else if (g.out_row >= 0) {
        out = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_o_off) +
              ((size_t)g.out_row * kHeads + h) * kDv;
        out_lse = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_lse_off) + (size_t)g.out_row * kHeads + h;
      } else {
        out = p.o_parts + ((size_t)g.u * kHeads + h) * kDv;
        out_lse = p.lses + (size_t)g.u * kHeads + h;
      }
      out += 256 * rank + 128 * e;
      uint32_t ov[32];
      __syncwarp();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem + lane_off + kColO + 128 * e + 32 * c, ov);
        tmem_wait_ld();
        float4* o4 = reinterpret_cast<float4*>(out + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o4[i] = make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                              __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
      }
      // A piece's LSE is written by both CTAs of the pair (the same value:
      // both computed the same scores and sums), so that each CTA's own count
      // below covers every LSE its merge reads.
      if (e == 0 && out_lse && (rank == 0 || piece))
        *out_lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      tc_fence_before();
      gt += nt;
      ++n_epi;
      if (piece && gr.pieces <= kMlaMergeInKernel) {
        // count this CTA's piece once all its rows are out (every thread's
        // stores, then a fence, then its arrival); the count that completes
        // the group merges it. Bounded waits on mbarriers, not bar.sync, so
        // that an abort cannot leave threads waiting for one that left.
        __threadfence();
        bar_arrive(bar(BPC));
        if (threadIdx.x == 0) {
          int last = 0;
          if (wait_bar(bar(BPC), n_pc & 1u, abort_flag, p.err, false)) {
            __threadfence();
            GroupRec* grw = reinterpret_cast<GroupRec*>(const_cast<char*>(p.ws) + p.L.grp_off);
            last = atomicAdd(&grw[g.b].cnt[rank], 1) == gr.pieces - 1 ? 1 : 0;
            __threadfence();
          }
          *merge_flag = last;
          bar_arrive(bar(BGO));
        }
        if (!wait_warp(bar(BGO), n_pc & 1u, abort_flag, p.err, false)) break;
        ++n_pc;
        if (*merge_flag) {
          __threadfence();
          merge_pieces(p, g.b, gr.tmp_begin, gr.pieces, rank, warp, lane,
                       reinterpret_cast<float*>(smem + Lay::kOffMw));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
  }
  cluster_sync();  // neither CTA exits while the other's copies or arrivals may still reach it
}

// One-call path, after the attention kernel: the row groups of the plan's
// finish list -- no token in any shard (o = 0, LSE = -inf), or cut into more
// than kMlaMergeInKernel pieces -- one warp per output row over the whole GPU:
// lane k holds the LSEs of pieces k, k + 32, ... (a group has at most one
// piece per CTA pair, at most 128: the launch checks), the weights follow by
// warp reductions, and each lane accumulates 16 of the row's 512 columns,
// four pieces per round of loads.
constexpr int kFinishThreads = 256;
constexpr int kFinishMax = 128;

__global__ void __launch_bounds__(kFinishThreads) mla_finish_kernel(const char* __restrict__ ws, WsLayout L,
                                                                     float* __restrict__ o,
                                                                     float* __restrict__ lse_out) {
  const int n_fin = reinterpret_cast<const WsHeader*>(ws)->n_finish;
  const int* fin = reinterpret_cast<const int*>(ws + L.fin_off);
  const GroupRec* grp = reinterpret_cast<const GroupRec*>(ws + L.grp_off);
  const float* tmp_o = reinterpret_cast<const float*>(ws + L.tmp_o_off);
  const float* tmp_lse = reinterpret_cast<const float*>(ws + L.tmp_lse_off);
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)n_fin * kHeads;
  const long long warps = (long long)gridDim.x * (kFinishThreads / 32);
  for (long long x = (long long)blockIdx.x * (kFinishThreads / 32) + (threadIdx.x >> 5); x < rows; x += warps) {
    const int rg = fin[x / kHeads], h = (int)(x % kHeads);
    const GroupRec gr = grp[rg];
    const int n = gr.pieces;
    float l[kFinishMax / 32], w[kFinishMax / 32];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kFinishMax / 32; ++c) {
      const int k = lane + 32 * c;
      l[c] = k < n ? __ldcg(tmp_lse + (size_t)(gr.tmp_begin + k) * kHeads + h) : -INFINITY;
      M = fmaxf(M, l[c]);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    float wsum = 0.f;
#pragma unroll
    for (int c = 0; c < kFinishMax / 32; ++c) {
      w[c] = (M == -INFINITY || l[c] == -INFINITY) ? 0.f : expf(l[c] - M);
      wsum += w[c];
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, s);
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int k0 = 0; k0 < n; k0 += 4) {  // (k0 .. k0 + 3 lie in one group of 32)
      const int c = k0 >> 5;
      const float wc = c == 0 ? w[0] : c == 1 ? w[1] : c == 2 ? w[2] : w[3];
      float4 v[4][4];
      float wk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + u;
        wk[u] = __shfl_sync(0xffffffffu, wc, k & 31);
        if (k < n) {
          const float4* src = reinterpret_cast<const float4*>(tmp_o + ((size_t)(gr.tmp_begin + k) * kHeads + h) * kDv);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[u][j] = __ldcg(src + lane + 32 * j);
        } else {
          wk[u] = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) v[u][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          acc[j] = make_float4(fmaf(wk[u], v[u][j].x, acc[j].x), fmaf(wk[u], v[u][j].y, acc[j].y),
                               fmaf(wk[u], v[u][j].z, acc[j].z), fmaf(wk[u], v[u][j].w, acc[j].w));
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float4* dst = reinterpret_cast<float4*>(o + ((size_t)rg * kHeads + h) * kDv);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[lane + 32 * j] = make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
    if (lane == 0 && lse_out) lse_out[(size_t)rg * kHeads + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Token-split pair kernel (bf16 cache)
// ---------------------------------------------------------------------------
// The same results as mla_partial_kernel<false>, with a page's work divided
// differently between the two CTAs of the pair. CTA r still accumulates value
// dims [256 r, 256 r + 256) of O, but scores only its own 32 tokens of each
// 64-token page (tokens 32 r .. 32 r + 31): S_r = Q . K_r^T (M = 128, N = 32,
// K = 576). The row maxima of the two halves and the two halves of P are
// exchanged through distributed shared memory, and each CTA's P.V runs over
// all 64 tokens. A CTA then holds only what it reads: its own 32 tokens in
// full (for its score) plus the other 32 tokens' rows of its own value dims
// (for P.V) -- 52 KB per page, 56 KB with its P_lo, instead of 72 KB -- so
// three stages fit where two did, and each SM takes in 52 KB per page
// instead of 72. (The score itself is barely cheaper: on this part a
// tcgen05 MMA of M = 128, K = 16 takes ~37 cycles for any N up to 64, so 36
// MMAs of N = 32 cost about what 36 of N = 64 do; the gain is the deeper
// pipeline.) Per page and CTA:
//   1. the copies (three TMA copies): its own tokens' other value dims, which
//      the other CTA needs for P.V (one multicast copy into both CTAs, at
//      the same slots), its own tokens' value dims, dims 512-575; plus the
//      other CTA's multicast of its tokens' rows of this CTA's value dims
//   2. S_r into TMEM (query dims 0-447 as the A operand in TMEM, 448-575 in
//      shared memory)
//   3. the row maximum of the own 32 tokens, sent to the other CTA (st.async
//      stores that complete on its barrier); both then take the maximum of
//      the two halves and run the same lazy rescale, so their running maxima
//      stay equal without further talk
//   4. P of the own tokens as two bf16 terms (hi, lo) into the slots only the
//      score read; hi goes to the other CTA with one bulk copy, lo only when
//      a tile carries a noticeable share of some row's weight (a flag tells
//      the other CTA, whose lo buffer is a single slot it releases after use)
//   5. O_r += P . V_r over both token halves
// At the end of an output row group the two CTAs' row sums are exchanged the
// same way. The waits that other warps' progress ends suspend (try_wait):
// eleven warps share four schedulers, and polling warps took issue slots
// from the softmax warps (512-sequence step 14.4 -> 12.4 ms). Two are
// polled: the producer's wait for a free stage and the score warp's, so that
// the copy and the score leave at once. The score of tile g also waits until
// the P.V of tile g - 2 is in the tensor pipe, which runs MMAs in issue
// order: that P.V frees the stage the copy of tile g + 1 needs. Every wait is
// bounded, as in mla_partial_kernel.
namespace ts {
constexpr int kStages = 3;
constexpr int kHalf = 32;                          // tokens of a page per CTA
constexpr int kBox = kHalf * 128;                  // 64 columns x 32 rows of bf16: 4 KB
constexpr int kSlots = 14;                         // boxes per stage
constexpr int kStage = kSlots * kBox;              // 56 KB
// slots of a stage: 0-3 tokens 0-31 x dims 256-511 (copied by CTA 0 into
// both), 4-7 tokens 32-63 x dims 0-255 (copied by CTA 1 into both), 8-11 the
// own tokens x the own value dims, 12 the own tokens x dims 512-575, 13 spare.
// After the score, CTA r's slots 4r .. 4r + 3 hold P_hi (two token halves of
// 8 KB: its own and the other CTA's) and slots 12-13 its own P_lo.
constexpr int kSlotOwnV = 8, kSlotRope = 12, kSlotLo = 12;
constexpr int kPHalf = kHeads * kHalf * 2;         // 8 KB: 128 heads x 32 tokens of bf16
constexpr int kKStepsTmem = 28;                    // query dims 0-447 in TMEM
constexpr int kQChunks = 2;                        // query dims 448-575 in shared memory
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 288;  // 256 + 32 + 224 columns
constexpr int kOffKv = 0;
constexpr int kOffQ = kOffKv + kStages * kStage;
constexpr int kOffLoPeer = kOffQ + kQChunks * kQChunkBytes;  // the other CTA's P_lo half
constexpr int kOffBar = kOffLoPeer + kPHalf;
constexpr int kNumBars = 40;
constexpr int kOffMisc = kOffBar + kNumBars * 8;   // TMEM slot, abort, merge flag, P flags, lo votes, counters, block ring
constexpr int kOffMx = kOffMisc + 256;             // [stage][head]: the other CTA's row maxima
constexpr int kOffLx = kOffMx + kStages * kHeads * 4;  // [2][head]: row-sum halves of this CTA
constexpr int kOffLp = kOffLx + 2 * kHeads * 4;        // [2][head]: the other CTA's row sums
constexpr int kOffMw = kOffLp + 2 * kHeads * 4;        // merge weights
constexpr int kSmemBytes = kOffMw + kSoftmaxWarps * 16 * kMlaMergeInKernel * 4 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kStage % 1024 == 0 && kOffQ % 1024 == 0 && kOffLoPeer % 1024 == 0, "swizzle atoms");
constexpr int B_QFULL = 0, B_QEMPTY = 1, B_QT = 2, B_SFULL = 3, B_SEMPTY = 4, B_LOFREE = 5, B_DRAIN = 6,
              B_DRAIN2 = 7, B_PC = 8, B_GO = 9, B_XCH = 10 /* + quadrant */, B_LX = 14 /* + parity */,
              B_KVFULL = 16, B_KVEMPTY = B_KVFULL + kStages, B_MX = B_KVEMPTY + kStages,
              B_POWN = B_MX + kStages, B_PPEER = B_POWN + kStages, B_PEMPTY = B_PPEER + kStages,
              B_PLO = B_PEMPTY + kStages;  // the other CTA's P_lo half landed
static_assert(B_PLO + 1 <= kNumBars, "barrier slots");

// slot of 64-column box c (0-8) of CTA r's own tokens
__device__ __forceinline__ int score_slot(int c, int r) {
  return c == 8 ? kSlotRope : (c >> 2) == r ? kSlotOwnV + (c & 3) : 4 * r + (c & 3);
}
// first slot of the value rows of token half h for CTA r
__device__ __forceinline__ int value_slot(int h, int r) { return h == r ? kSlotOwnV : 4 * h; }
// byte offset of 8-token chunk `chunk` of row `row` in a 128-row x 32-token
// K-major tile with the 64-byte swizzle: 64-byte rows, the 16-byte chunk
// index XORed with address bits 7-8 (= (row / 2) % 4)
__device__ __forceinline__ uint32_t ptile_off(int row, int chunk) {
  return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}
}  // namespace ts

// Four consecutive 64-column boxes (column blocks z .. z + 3) of 32 rows from
// y, landing as four consecutive 4 KB boxes (the 3-D map's innermost dims are
// the 64 columns and the rows, its outer dim the column block)
__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap* map, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(z), "r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load4_mc(uint32_t dst, const CUtensorMap* map, int y, int z, uint32_t bar,
                                             uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;\n"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(z), "r"(bar), "h"(cta_mask) : "memory");
}
// the same shared-memory offset in CTA `peer` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(peer));
  return r;
}
// 4-byte store into another CTA's shared memory that completes as tx bytes
// on that CTA's mbarrier (no fence or arrival needed by the sender)
__device__ __forceinline__ void st_async_u32(uint32_t a, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];\n" ::"r"(a), "r"(v), "r"(bar)
               : "memory");
}
// bulk copy from this CTA's shared memory into another CTA's (dst and bar are
// cluster addresses), completing on that CTA's mbarrier
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
               ::"r"(dst), "r"(src), "r"(bytes), "r"(bar) : "memory");
}
// bounded, warp-uniform wait with cluster-scope acquire (the phase may have
// been completed by the other CTA). It suspends in try_wait instead of
// polling: eleven warps share four schedulers here, and polling warps take
// issue slots from the softmax warps (measured: 14.38 -> 12.36 ms on the
// 512-sequence step).
__device__ __forceinline__ bool wait_warp_cluster(uint32_t b, uint32_t parity, volatile int* abort_flag,
                                                  int32_t* err) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (__all_sync(0xffffffffu, bar_try_cluster(b, parity))) return true;
    if ((i & 63u) == 63u && __any_sync(0xffffffffu, *abort_flag != 0)) return false;
  }
  *abort_flag = 1;
  raise_flag(err, DCP_DEVERR_TIMEOUT);
  return false;
}
// bounded wait of one thread that polls (test_wait) instead of suspending
__device__ __forceinline__ bool poll_bar(uint32_t b, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (bar_test(b, parity)) return true;
    if ((i & 63u) == 63u && *abort_flag) return false;
  }
  *abort_flag = 1;
  raise_flag(err, DCP_DEVERR_TIMEOUT);
  return false;
}
// K-major shared-memory descriptor, 64-byte swizzle: 64-byte rows, 8-row
// groups 512 B apart (a 128-row x 32-token bf16 tile)
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)(512 >> 4) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 4ull << 61;  // 64-byte swizzle
  return d;
}
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ MlaParams p) {
  using namespace ts;
  // (the names this kernel shares with mla_partial_kernel's constants)
  constexpr int kStages = ts::kStages, kOffKv = ts::kOffKv, kKStepsTmem = ts::kKStepsTmem;
  constexpr uint32_t kColO = ts::kColO, kColS = ts::kColS, kColQ = ts::kColQ;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = saddr(smem);
  const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  auto stage_base = [&](uint32_t s) { return sbase + kOffKv + s * kStage; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  volatile int* pflag = reinterpret_cast<volatile int*>(smem + kOffMisc + 16);     // [stage]: the other CTA's lo
  volatile int* lo_votes = reinterpret_cast<volatile int*>(smem + kOffMisc + 32);  // [stage][softmax warp]
  volatile int* pv_issued = reinterpret_cast<volatile int*>(smem + kOffMisc + 128);  // P.V tiles issued
  // each tile's physical block as the producer read it (ring of 16), so that
  // the softmax warps need no block-table load of their own
  volatile int* phys_written = reinterpret_cast<volatile int*>(smem + kOffMisc + 136);
  volatile int* phys_ring = reinterpret_cast<volatile int*>(smem + kOffMisc + 160);

  if (threadIdx.x == 0) {
    bar_init(bar(B_QFULL), kSoftmaxThreads);
    bar_init(bar(B_QEMPTY), 1);
    bar_init(bar(B_QT), 1);
    bar_init(bar(B_SFULL), 1);
    bar_init(bar(B_SEMPTY), kSoftmaxThreads);
    bar_init(bar(B_LOFREE), 1);  // the other CTA's P.V finished with this CTA's lo in its buffer
    bar_init(bar(B_DRAIN), 1);
    bar_init(bar(B_DRAIN2), 1);
    bar_init(bar(B_PC), kSoftmaxThreads);
    bar_init(bar(B_GO), 1);
    for (int q4 = 0; q4 < 4; ++q4) bar_init(bar(B_XCH + q4), 64);
    for (int x = 0; x < 2; ++x) bar_init(bar(B_LX + x), 1);  // the other CTA's row sums (512 bytes)
    bar_init(bar(B_PLO), 1);
    for (int s = 0; s < kStages; ++s) {
      bar_init(bar(B_KVFULL + s), 1);
      bar_init(bar(B_KVEMPTY + s), 2);           // both CTAs' P.V of the page
      bar_init(bar(B_MX + s), 1);                // the other CTA's row maxima (512 bytes)
      bar_init(bar(B_POWN + s), kSoftmaxThreads);
      bar_init(bar(B_PPEER + s), 1);             // the other CTA's P_hi half and lo flag landed
      bar_init(bar(B_PEMPTY + s), 1);
    }
    *abort_flag = 0;
    *pv_issued = 0;
    *phys_written = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(saddr(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either writes into the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int* cta_begin = reinterpret_cast<const int*>(p.ws + p.L.cta_off);
  const int k_begin = cta_begin[cluster], k_end = cta_begin[cluster + 1];
  auto n_tiles = [&](int k) {
    const ItemRec it = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k];
    return it.t1 - it.t0;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t fills = 0;
    int q_done = 0;
    bool stop = false;
    for (int k = k_begin; k < k_end && !stop; ++k) {
      const ItemGeom g = item_geom(p, k);
      const int nt = g.t1 - g.t0;
      const bool same_q = same_rows(p, k, k_begin);
      if (lane == 0 && rank == 0 && k + 1 < k_end && !same_rows(p, k + 1, k_begin)) {
        const int nb = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k + 1].lane % p.B;
        l2_prefetch(p.q + (size_t)nb * kHeads * kDk, kHeads * kDk * 2);
      }
      int cur = lane < nt ? tile_block(p, g, g.t0 + lane) : -1;
      int nxt = 32 + lane < nt ? tile_block(p, g, g.t0 + 32 + lane) : -1;
      bool ok = true;
      if (lane == 0 && !same_q) {
        if (q_done > 0 && !wait_bar(bar(B_QEMPTY), (q_done - 1) & 1, abort_flag, p.err, false)) {
          ok = false;
        } else {
          bar_arrive_tx(bar(B_QT), kQChunks * kQChunkBytes);
          for (int c = 0; c < kQChunks; ++c)
            tma_load(sbase + kOffQ + c * kQChunkBytes, &p.tm_q, 448 + 64 * c, g.b * kHeads, bar(B_QT));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) { stop = true; break; }
      if (!same_q) ++q_done;
      for (int j = 0; j < nt; ++j) {
        if ((j & 31) == 0 && j > 0) {
          cur = nxt;
          nxt = j + 32 + lane < nt ? tile_block(p, g, g.t0 + j + 32 + lane) : -1;
        }
        const int phys = __shfl_sync(0xffffffffu, cur, j & 31);
        int phys_pf = -1;
        if (kPrefetch > 0) {
          const int jp = j + kPrefetch;
          const int a = __shfl_sync(0xffffffffu, cur, jp & 31), b2 = __shfl_sync(0xffffffffu, nxt, jp & 31);
          phys_pf = jp < nt ? ((jp >> 5) == (j >> 5) ? a : b2) : -1;
        }
        if (lane == 0) {
          const uint32_t s = fills % kStages, use = fills / kStages;
          // (polled: the copy should leave as soon as both P.V have freed the stage)
          if (use > 0 && !poll_bar(bar(B_KVEMPTY + s), (use - 1) & 1u, abort_flag, p.err)) {
            ok = false;
          } else {
            phys_ring[fills & 15u] = phys;
            __threadfence_block();
            *phys_written = (int)fills + 1;
            if (phys < 0 && rank == 0) raise_flag(p.err, DCP_DEVERR_BLOCK_RANGE);
            // rows of this CTA's tokens (an unusable entry reads zeros above row 0)
            const int row = (phys < 0 ? -kTile : phys * kTile) + kHalf * (int)rank;
            const uint32_t st = stage_base(s);
            // 13 boxes land here: 5 private, 4 of this CTA's multicast, 4 of the other's
            bar_arrive_tx(bar(B_KVFULL + s), 13 * kBox);
            // the other CTA's value dims of the own tokens (into both CTAs), the
            // own value dims, dims 512-575
            tma_load4_mc(st + 4 * rank * kBox, &p.tm_kv4[g.shard], row, 4 * (int)peer, bar(B_KVFULL + s), 0x3);
            tma_load4(st + kSlotOwnV * kBox, &p.tm_kv4[g.shard], row, 4 * (int)rank, bar(B_KVFULL + s));
            tma_load(st + kSlotRope * kBox, &p.tm_kv[g.shard], 512, row, bar(B_KVFULL + s));
            if (kPrefetch > 0 && rank == 0 && phys_pf >= 0)
              l2_prefetch(static_cast<const char*>(p.sh.k[g.shard]) + (size_t)phys_pf * kStageBytes, kStageBytes);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) { stop = true; break; }
        ++fills;
      }
    }
    if (lane == 0 && *abort_flag) {  // copies in flight must land before the CTA may exit
      if (q_done > 0) drain_bar(bar(B_QT), (q_done - 1) & 1u);
      const uint32_t f0 = fills > (uint32_t)kStages ? fills - kStages : 0;
      for (uint32_t f = f0; f < fills + 1; ++f) drain_bar(bar(B_KVFULL + f % kStages), (f / kStages) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ score MMA issuer
    const uint32_t id_s = idesc(128, kHalf, 0);
    const uint64_t qdesc0 = sdesc(sbase + kOffQ, 0);
    int ks = k_begin, js = 0, nts = ks < k_end ? n_tiles(ks) : 0;
    uint32_t g_s = 0, q_loads = 0;
    bool q_ready = false;
    uint32_t idle = 0;
    while (ks < k_end) {
      bool progressed = false;
      if (!q_ready && bar_test_warp(bar(B_QFULL), q_loads & 1u) && bar_test_warp(bar(B_QT), q_loads & 1u)) {
        q_ready = true;
        tc_fence_after();
      }
      const uint32_t s = g_s % kStages;
      // The score of tile g waits until the P.V of tile g - 2 is in the tensor
      // pipe (which runs MMAs in issue order): that P.V frees the stage the
      // copy of tile g + 1 needs, while the score has a tile of slack.
      if (q_ready && (g_s < 2 || *pv_issued >= (int)g_s - 1) && bar_test_warp(bar(B_KVFULL + s), (g_s / kStages) & 1u) &&
          (g_s == 0 || bar_test_warp(bar(B_SEMPTY), (g_s - 1) & 1u))) {
        tc_fence_after();
        const uint64_t kd = sdesc(stage_base(s), 0);
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
          const int box = kk >> 2;
          const uint64_t bdesc = kd + (uint64_t)((score_slot(box, (int)rank) * kBox + 32 * (kk & 3)) >> 4);
          if (kk < kKStepsTmem) {
            mma_ts(tmem + kColS, tmem + kColQ + 8 * kk, bdesc, id_s, kk > 0);
          } else {
            const int qk = kk - kKStepsTmem;
            mma_ss(tmem + kColS, qdesc0 + (uint64_t)((((qk >> 2) * kQChunkBytes) + 32 * (qk & 3)) >> 4), bdesc, id_s,
                   1);
          }
        }
        mma_commit(bar(B_SFULL));
        if (++js == nts) {
          if (!(ks + 1 < k_end && same_rows(p, ks + 1, k_begin))) {
            mma_commit(bar(B_QEMPTY));
            ++q_loads;
            q_ready = false;
          }
          ++ks;
          js = 0;
          nts = ks < k_end ? n_tiles(ks) : 0;
        }
        ++g_s;
        progressed = true;
      }
      if (progressed) {
        idle = 0;
      } else if (++idle >= kSpinLimit) {
        *abort_flag = 1;
        raise_flag(p.err, DCP_DEVERR_TIMEOUT);
        break;
      } else if ((idle & 63u) == 0 && __any_sync(0xffffffffu, *abort_flag != 0)) {
        break;
      }
    }
    mma_commit(bar(B_DRAIN));
    drain_bar(bar(B_DRAIN), 0);
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P exchange and P.V MMA issuer
    const uint32_t id_pv = idesc(128, 256, 1);
    int kp = k_begin, jp = 0, ntp = kp < k_end ? n_tiles(kp) : 0;
    bool acc_in = false;
    uint32_t g_p = 0, lo_sent = 0, lo_recv = 0;
    bool ok = true;
    while (kp < k_end && ok) {
      const uint32_t s = g_p % kStages, ph = (g_p / kStages) & 1u;
      const uint32_t st = stage_base(s);
      const uint32_t pbase = st + 4 * rank * kBox;  // P_hi: token half h at pbase + h * kPHalf
      // 0. expect the other CTA's P_hi half and flag for this tile
      if (lane == 0) bar_arrive_tx(bar(B_PPEER + s), kPHalf + 4);
      // 1. this CTA's P is in place
      if (!wait_warp_cluster(bar(B_POWN + s), ph, abort_flag, p.err)) { ok = false; break; }
      int f_own = 0;
#pragma unroll
      for (int w = 0; w < kSoftmaxWarps; ++w) f_own |= lo_votes[kSoftmaxWarps * s + w];
      // 2. send it: hi always, lo when asked for (into the other CTA's single
      // lo buffer, once its P.V has finished with the previous one)
      if (f_own && lo_sent > 0 && !wait_warp_cluster(bar(B_LOFREE), (lo_sent - 1) & 1u, abort_flag, p.err)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t pb = peer_addr(bar(B_PPEER + s), peer);
        // the other CTA keeps its P_hi in its slots 4 peer ..; this half goes to token half `rank`
        bulk_to_peer(peer_addr(st + 4 * peer * kBox + rank * kPHalf, peer), pbase + rank * kPHalf, kPHalf, pb);
        st_async_u32(peer_addr(sbase + kOffMisc + 16 + 4 * s, peer), (uint32_t)f_own, pb);
        if (f_own)
          bulk_to_peer(peer_addr(sbase + kOffLoPeer, peer), st + kSlotLo * kBox, kPHalf, peer_addr(bar(B_PLO), peer));
      }
      __syncwarp();
      if (f_own) ++lo_sent;
      // 3. the other CTA's half (and its lo, when its flag asks for it)
      if (!wait_warp_cluster(bar(B_PPEER + s), ph, abort_flag, p.err)) { ok = false; break; }
      const int f_peer = pflag[s];
      if (f_peer) {
        if (lane == 0) bar_arrive_tx(bar(B_PLO), kPHalf);
        __syncwarp();
        if (!wait_warp_cluster(bar(B_PLO), lo_recv & 1u, abort_flag, p.err)) { ok = false; break; }
        ++lo_recv;
      }
      tc_fence_after();
      // 4. O_r += P . V_r over the two token halves
      bool first = jp == 0 && !acc_in;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t vd = sdesc(st + value_slot(h, (int)rank) * kBox, kBox);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          mma_ss(tmem + kColO, sdesc_sw64(pbase + h * kPHalf + 32 * kk),
                 vd + (uint64_t)((2048 * kk) >> 4), id_pv, first ? 0 : 1);
          first = false;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool own = h == (int)rank;
        if (!(own ? f_own : f_peer)) continue;
        const uint32_t lo_tile = own ? st + kSlotLo * kBox : sbase + kOffLoPeer;
        const uint64_t vd = sdesc(st + value_slot(h, (int)rank) * kBox, kBox);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_ss(tmem + kColO, sdesc_sw64(lo_tile + 32 * kk), vd + (uint64_t)((2048 * kk) >> 4),
                 id_pv, 1);
      }
      mma_commit_mc(bar(B_KVEMPTY + s), 0x3);  // the stage is free in both CTAs once both P.V finished
      mma_commit(bar(B_PEMPTY + s));
      if (lane == 0) *pv_issued = (int)g_p + 1;
      if (f_peer) {
        mma_commit_mc(bar(B_LOFREE), (uint16_t)(1u << peer));  // the other CTA may send its next lo
      }
      if (++jp == ntp) {
        ++kp;
        jp = 0;
        ntp = kp < k_end ? n_tiles(kp) : 0;
        acc_in = kp < k_end && continues(p, kp, k_begin);
      }
      ++g_p;
    }
    if (!ok && lane == 0) {
      // the other CTA's copies into this one may still be in flight: let the
      // ones it can have issued land (bounded polls)
      for (uint32_t f = g_p; f < g_p + kStages; ++f) drain_bar(bar(B_PPEER + f % kStages), (f / kStages) & 1u);
      drain_bar(bar(B_PLO), lo_recv & 1u);
    }
    __syncwarp();
    mma_commit(bar(B_DRAIN2));
    drain_bar(bar(B_DRAIN2), 0);
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // Warp w: TMEM lane quadrant qd = w % 4 (heads 32 qd ..), half e = w / 4:
    // the own tokens 16 e .. 16 e + 15 for the exponentials and P, and this
    // CTA's value dims 128 e .. 128 e + 127 of O. Both warps of a quadrant read
    // all 32 own scores of their rows, so they take the same maximum.
    const int qd = warp & 3, e = warp >> 2;
    const int h = 32 * qd + lane;
    const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
    const bool pos_scale = p.sl2 >= 0.f;
    float* lx = reinterpret_cast<float*>(smem + kOffLx);
    const float* mxp = reinterpret_cast<const float*>(smem + kOffMx);
    const float* lp = reinterpret_cast<const float*>(smem + kOffLp);
    uint32_t gt = 0;
    int n_q = 0, n_epi = 0;
    uint32_t n_pc = 0;
    float m_run = -INFINITY, l_half = 0.f;
    bool ok = true;
    for (int k = k_begin; k < k_end && ok; ++k) {
      const ItemGeom g = item_geom(p, k);
      const int nt = g.t1 - g.t0;
      if (!same_rows(p, k, k_begin)) {
        // query dims 224 e .. 224 e + 223 into TMEM, after the previous row group's score MMAs
        if (n_q > 0 && !wait_warp(bar(B_QEMPTY), (n_q - 1) & 1, abort_flag, p.err, false)) break;
        tc_fence_after();
        const uint4* qr = reinterpret_cast<const uint4*>(p.q + ((size_t)g.b * kHeads + h) * kDk + 224 * e);
        uint32_t qv[16];
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < 7; ++c) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = qr[4 * c + i];
            qv[4 * i] = v.x;
            qv[4 * i + 1] = v.y;
            qv[4 * i + 2] = v.z;
            qv[4 * i + 3] = v.w;
          }
          tmem_st16(tmem + lane_off + kColQ + 112 * e + 16 * c, qv);
        }
        tmem_wait_st();
        tc_fence_before();
        bar_arrive(bar(B_QFULL));
        ++n_q;
      }
      if (!continues(p, k, k_begin)) {
        m_run = -INFINITY;
        l_half = 0.f;
      }
      for (int j = 0; j < nt; ++j) {
        const uint32_t gi = gt + j, s = gi % kStages, ph = (gi / kStages) & 1u;
        const uint32_t st = stage_base(s);
        const int t = g.t0 + j;
        int phys = -2;  // the tile's block, as the producer published it
        for (uint32_t it = 0; it < kSpinLimit; ++it) {
          if (*phys_written > (int)gi) { phys = phys_ring[gi & 15u]; break; }
          if ((it & 63u) == 63u && *abort_flag) break;
        }
        if (phys == -2) {
          if (!*abort_flag) { *abort_flag = 1; raise_flag(p.err, DCP_DEVERR_TIMEOUT); }
          ok = false;
          break;
        }
        const int n_valid = phys < 0 ? 0 : min(kTile, g.hi - (g.lo + kTile * t));
        const int own0 = kHalf * (int)rank;  // first own token of the tile
        // 1. the own 32 scores (polled: a suspended wait wakes late)
        if (!wait_warp_cluster(bar(B_SFULL), gi & 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + kColS, sv);
        tmem_wait_ld();
        tc_fence_before();
        bar_arrive(bar(B_SEMPTY));
        // 2. the own maximum (of scale * s, as scale * max or min of s), sent
        float raw_ext = pos_scale ? -INFINITY : INFINITY;
        if (n_valid - own0 >= kHalf) {  // common case: no masking; a tree of three-input extrema
          raw_ext = pos_scale ? ext_tree<32, true>(sv) : ext_tree<32, false>(sv);
        } else {
#pragma unroll
          for (int i = 0; i < kHalf; ++i) {
            const float x = __uint_as_float(sv[i]);
            if (own0 + i < n_valid) raw_ext = pos_scale ? fmaxf(raw_ext, x) : fminf(raw_ext, x);
          }
        }
        const float mx_own = n_valid > own0 ? raw_ext * p.sl2 : -INFINITY;
        if (threadIdx.x == 0) bar_arrive_tx(bar(B_MX + s), kHeads * 4);  // expect the other CTA's maxima
        if (e == 0)
          st_async_u32(peer_addr(sbase + kOffMx + (s * kHeads + h) * 4, peer), __float_as_uint(mx_own),
                       peer_addr(bar(B_MX + s), peer));
        if (!wait_warp_cluster(bar(B_MX + s), ph, abort_flag, p.err)) { ok = false; break; }
        const float mx = fmaxf(mx_own, mxp[s * kHeads + h]);
        float m_new = m_run, alpha = 1.f;
        bool rescale = false;
        if (m_run == -INFINITY) {
          m_new = mx;
        } else if (mx > m_run + kRescaleThreshold) {
          m_new = mx;
          alpha = exp2f(m_run - m_new);
          rescale = true;
        }
        const float ref = m_new == -INFINITY ? 0.f : m_new;
        // 3. P of this warp's 16 own tokens
        float sc[16];
        float lsum;
        {
          uint32_t mine[16];  // this warp's 16 scores (static register indices)
          if (e == 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) mine[i] = sv[i];
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) mine[i] = sv[16 + i];
          }
          // two scores scaled and shifted per instruction; the row sum in pairs
          const int tok0 = own0 + 16 * e;
          const unsigned long long s2 = f2pack(p.sl2, p.sl2), r2 = f2pack(-ref, -ref);
          unsigned long long a0 = f2pack(0.f, 0.f), a1 = a0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(mine[2 * i]), __uint_as_float(mine[2 * i + 1])), s2, r2), x0, x1);
            sc[2 * i] = tok0 + 2 * i < n_valid ? ex2_ftz(x0) : 0.f;
            sc[2 * i + 1] = tok0 + 2 * i + 1 < n_valid ? ex2_ftz(x1) : 0.f;
            if (i & 1)
              a1 = fadd2(a1, f2pack(sc[2 * i], sc[2 * i + 1]));
            else
              a0 = fadd2(a0, f2pack(sc[2 * i], sc[2 * i + 1]));
          }
          float y0, y1;
          f2unpack(fadd2(a0, a1), y0, y1);
          lsum = y0 + y1;
        }
        l_half = l_half * alpha + lsum;
        m_run = m_new;
        // A warp's running sum covers a quarter of its rows' tokens here (half in
        // mla_partial_kernel), so twice the fraction asks, typically, for the
        // same share of the row; a skipped tile's share of the row stays below
        // 1/16, and dropping its residual changes O by at most 2^-9 x 1/16 x
        // max|v|.
        const bool any_lo = __any_sync(0xffffffffu, lsum > 2.f * kLoFraction * l_half);
        {
          const uint32_t hi_tile = st + 4 * rank * kBox + rank * kPHalf, lo_tile = st + kSlotLo * kBox;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) split_p_bf16(sc[8 * c + 2 * k2], sc[8 * c + 2 * k2 + 1], hi[k2], lo[k2]);
            const uint32_t off = ptile_off(h, 2 * e + c);
            st_shared_v4(hi_tile + off, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(lo_tile + off, lo[0], lo[1], lo[2], lo[3]);
          }
          if (lane == 0) lo_votes[kSoftmaxWarps * s + warp] = any_lo ? 1 : 0;
        }
        // 4. value rows past the end of a partial tile may hold anything: zero
        // this CTA's value dims of those rows, in both token halves
        if (n_valid < kTile) {
          const int tid = threadIdx.x;
          for (int x = tid; x < (kTile - n_valid) * 4 * 8; x += kSoftmaxThreads) {
            const int tok = n_valid + x / 32, c = (x >> 3) & 3, piece = x & 7;
            const int hh = tok / kHalf, r = tok % kHalf;
            st_shared_v4(st + (value_slot(hh, (int)rank) + c) * kBox + r * 128 + piece * 16, 0u, 0u, 0u, 0u);
          }
        }
        // 5. lazy rescale of this warp's half of O, after the previous P.V
        if (__any_sync(0xffffffffu, rescale)) {
          if (gi >= 1 && !wait_warp(bar(B_PEMPTY + (gi - 1) % kStages), ((gi - 1) / kStages) & 1u, abort_flag, p.err,
                                    false)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t ov[32];
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            const uint32_t col = kColO + 128 * e + 32 * c;
            tmem_ld32(tmem + lane_off + col, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tmem + lane_off + col, ov);
          }
          tmem_wait_st();
        }
        // 6. publish P (for this CTA's P.V and for the copy to the other CTA)
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        tc_fence_before();
        bar_arrive(bar(B_POWN + s));
      }
      if (!ok) break;
      if (k + 1 < k_end && continues(p, k + 1, k_begin)) {
        gt += nt;
        continue;
      }
      // epilogue: this CTA's row sum (two halves), then the other CTA's
      lx[e * kHeads + h] = l_half;
      bar_arrive(bar(B_XCH + qd));
      if (!wait_warp(bar(B_XCH + qd), (uint32_t)n_epi & 1u, abort_flag, p.err, false)) break;
      const float l_cta = l_half + lx[(1 - e) * kHeads + h];
      const int px = n_epi & 1;
      if (threadIdx.x == 0) bar_arrive_tx(bar(B_LX + px), kHeads * 4);
      if (e == 0)
        st_async_u32(peer_addr(sbase + kOffLp + (px * kHeads + h) * 4, peer), __float_as_uint(l_cta),
                     peer_addr(bar(B_LX + px), peer));
      if (!wait_warp_cluster(bar(B_LX + px), ((uint32_t)n_epi >> 1) & 1u, abort_flag, p.err)) break;
      const float l_run = l_cta + lp[px * kHeads + h];
      const uint32_t glast = gt + nt - 1;
      if (!wait_warp(bar(B_PEMPTY + glast % kStages), (glast / kStages) & 1u, abort_flag, p.err, false)) break;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      float* out;
      float* out_lse;
      GroupRec gr;
      bool piece = false;
      if (p.o) {
        gr = reinterpret_cast<const GroupRec*>(p.ws + p.L.grp_off)[g.b];
        piece = gr.pieces > 1;
        if (piece) {
          const size_t row = (size_t)(gr.tmp_begin + cluster - gr.first_cta);
          out = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_o_off) + (row * kHeads + h) * kDv;
          out_lse = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_lse_off) + row * kHeads + h;
        } else {
          out = p.o + ((size_t)g.b * kHeads + h) * kDv;
          out_lse = p.lse_out ? p.lse_out + (size_t)g.b * kHeads + h : nullptr;
        }
      } else if (g.out_row >= 0) {
        out = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_o_off) +
              ((size_t)g.out_row * kHeads + h) * kDv;
        out_lse = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_lse_off) + (size_t)g.out_row * kHeads + h;
      } else {
        out = p.o_parts + ((size_t)g.u * kHeads + h) * kDv;
        out_lse = p.lses + (size_t)g.u * kHeads + h;
      }
      out += 256 * rank + 128 * e;
      uint32_t ov[32];
      __syncwarp();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem + lane_off + kColO + 128 * e + 32 * c, ov);
        tmem_wait_ld();
        float4* o4 = reinterpret_cast<float4*>(out + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o4[i] = make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                              __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
      }
      if (e == 0 && out_lse && (rank == 0 || piece))
        *out_lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      tc_fence_before();
      gt += nt;
      ++n_epi;
      if (piece && gr.pieces <= kMlaMergeInKernel) {
        __threadfence();
        bar_arrive(bar(B_PC));
        if (threadIdx.x == 0) {
          int last = 0;
          if (wait_bar(bar(B_PC), n_pc & 1u, abort_flag, p.err, false)) {
            __threadfence();
            GroupRec* grw = reinterpret_cast<GroupRec*>(const_cast<char*>(p.ws) + p.L.grp_off);
            last = atomicAdd(&grw[g.b].cnt[rank], 1) == gr.pieces - 1 ? 1 : 0;
            __threadfence();
          }
          *merge_flag = last;
          bar_arrive(bar(B_GO));
        }
        if (!wait_warp(bar(B_GO), n_pc & 1u, abort_flag, p.err, false)) break;
        ++n_pc;
        if (*merge_flag) {
          __threadfence();
          merge_pieces(p, g.b, gr.tmp_begin, gr.pieces, rank, warp, lane, reinterpret_cast<float*>(smem + kOffMw));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols));
  }
  cluster_sync();  // neither CTA exits while the other's copies or arrivals may still reach it
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 2-D bf16 map over rows of 576 latent/query columns; boxes of 64 columns
// (128 bytes, 128-byte swizzle) by box_rows rows; out-of-range rows read 0.
bool latent_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {576, rows};
  cuuint64_t strides[1] = {576 * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of the same rows for the token-split kernel: dims (64 columns,
// rows, 9 column blocks of 128 bytes), boxes of 64 columns x 32 rows x 4
// blocks, which land as four consecutive 4 KB boxes.
bool latent_map4(CUtensorMap* m, const void* base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, rows, 9};
  cuuint64_t strides[2] = {576 * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)ts::kHalf, 4};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Co-resident clusters on the current device for the bf16 (F8 = false) or
// the 8-bit kernel (0 on failure), cached.
template <bool F8>
int mla_clusters() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] > 0) return cache[dev];
  constexpr int kSmem = MlaLayout<F8>::kSmemBytes;
  if (cudaFuncSetAttribute(mla_partial_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess)
    return 0;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_partial_kernel<F8>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  cache[dev] = n;
  return n;
}

// Co-resident clusters of the token-split kernel (0 on failure), cached.
int mla_split_clusters() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] > 0) return cache[dev];
  if (cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ts::kSmemBytes) !=
      cudaSuccess)
    return 0;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = ts::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_split_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  cache[dev] = n;
  return n;
}

// The bf16 cache runs the token-split kernel (1) or the kernel that repeats
// the score in both CTAs (0).
#ifndef DCP_MLA_TOKEN_SPLIT
#define DCP_MLA_TOKEN_SPLIT 1
#endif
constexpr bool kTokenSplit = DCP_MLA_TOKEN_SPLIT != 0;

}  // namespace

int mla_ctas(const dcp_attn_desc& d, const DeviceInfo&) {
  if (d.kv_dtype == DCP_KV_FP8_E4M3) return mla_clusters<true>();
  return kTokenSplit ? mla_split_clusters() : mla_clusters<false>();
}

cudaError_t launch_mla(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                       float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas, int32_t* err,
                       cudaStream_t st, float* o, float* lse_out) {
  const bool f8 = d.kv_dtype == DCP_KV_FP8_E4M3;
  const bool split = !f8 && kTokenSplit;
  if (n_ctas <= 0 || (f8 ? mla_clusters<true>() : split ? mla_split_clusters() : mla_clusters<false>()) <= 0)
    return cudaErrorNotSupported;
  if (o && n_ctas > kFinishMax) return cudaErrorNotSupported;  // a row group's pieces must fit the finish kernel
  MlaParams p;
  memset(&p, 0, sizeof(p));
  if (!f8) {  // the 8-bit kernel copies its pages with plain bulk copies and loads its query itself
    if (!latent_map(&p.tm_q, q, (uint64_t)rs.B * kHeads, kHeads)) return cudaErrorNotSupported;
    for (int i = 0; i < rs.N; ++i) {  // boxes of a page (64 rows), or of a CTA's half page (32)
      if (!latent_map(&p.tm_kv[i], sh.k[i], (uint64_t)sh.nblk[i] * kTile, split ? ts::kHalf : kTile))
        return cudaErrorNotSupported;
      if (split && !latent_map4(&p.tm_kv4[i], sh.k[i], (uint64_t)sh.nblk[i] * kTile)) return cudaErrorNotSupported;
    }
  }
  p.sh = sh;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.ws = static_cast<const char*>(ws);
  p.L = L;
  p.o_parts = o_parts;
  p.lses = lses;
  p.o = o;
  p.lse_out = lse_out;
  p.err = err;
  p.B = rs.B;
  p.qlen = rs.qlen;
  p.sl2 = d.scale * kLog2e * (f8 ? d.k_scale : 1.f);
  p.v_scale = f8 ? d.v_scale : 1.f;
  if (f8)
    mla_partial_kernel<true><<<2 * n_ctas, kThreads, MlaLayout<true>::kSmemBytes, st>>>(p);
  else if (split)
    mla_split_kernel<<<2 * n_ctas, kThreads, ts::kSmemBytes, st>>>(p);
  else
    mla_partial_kernel<false><<<2 * n_ctas, kThreads, MlaLayout<false>::kSmemBytes, st>>>(p);
  if (o) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      return cudaErrorUnknown;
    // the list's length is on the device: a grid for up to ~4 rows per warp
    // at the 8-sequence size, and an immediate exit when the list is empty
    mla_finish_kernel<<<4 * sms, kFinishThreads, 0, st>>>(static_cast<const char*>(ws), L, o, lse_out);
  }
  return cudaGetLastError();
}

}  // namespace dcp
