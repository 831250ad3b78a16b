// Partial attention of many query rows per KV head (GQA, head dim 128) on
// the 5th-generation tensor cores (tcgen05 + TMEM + TMA) of sm_103a: the
// multi-token steps and prefill chunks whose query rows fill the 128 rows of
// the MMA.
//
// What it computes is step 2 of the method for every query token of the
// step (each shard attends the queries against its own KV slice only and
// emits a partial output plus LSE -- Qiita write-up "vLLMの-dcpが長文脈のKV
// キャッシュ重複を消して3倍速くする", section "トークンの区間でGPUに割り振る"),
// applied to the chunked / cached prefill of "Inference Systems
// Infrastructure Notes (7): DCP", section 4: query token j of sequence b sits
// at position seq_len - q_len + j and attends every token at or before it.
//
// Layout of the work: a lane is (shard, sequence, token group, KV head); its
// NB x 128 query rows are the NB*128/g tokens of the group times the g query
// heads of the KV head (row r = token slot r / g, head r % g), taken as NB
// blocks of 128 rows that share every K/V tile (NB = 2 once a step has 256
// rows per KV head: two groups of four softmax warps then work on the two
// blocks in turn while the tensor cores serve the other). The token groups of
// one (shard, sequence, KV head) read the same K/V; gangs of up to eight CTAs
// take consecutive groups over the same items (the union of their ranges;
// each row is masked at its own token), so the gang reads each tile at about
// the same time and L2 serves all but the first read. Per 64-token tile of
// the lane's range, for each block:
//   1. S = Q . K^T (M=128 rows, N=64 tokens, K=128) into TMEM, the queries
//      being the MMA's A operand in TMEM
//   2. online softmax per row (thread r owns TMEM lane r), causal at the
//      row's own token, in log2 units with the scale folded into one FMA per
//      score (a negative scale is taken as q -> -q, exact in bf16), lazy
//      rescale of O (only when the running max grows by more than 2^8)
//   3. P is written to shared memory as bf16, hi = bf16(p); where the tile
//      carries more than 1/32 of some row's running weight (the block's four
//      warps vote through an mbarrier) the residual lo = bf16(p - hi) is
//      written too and P_lo . V issued (elsewhere dropping it changes O by
//      at most 2^-9 x that share x max|v|)
//   4. O += P_hi . V (M=128, N=128, K=64) into TMEM, V being read by the MMA
//      straight from the copy of the tile (dims contiguous)
// TMA brings the K and V rows of a tile from the paged pools (boxes of
// min(block_size, 64) rows x 64 columns, 128-byte swizzle) into a 4-stage
// ring. One warp schedules the MMAs (non-blocking barrier polls, uniform
// control flow, one elect.sync-chosen lane issues); one warp copies; four
// warps per block run the softmax and the epilogue. Every barrier's phases are
// observed in order and never more than one phase late; every wait is
// bounded: on expiry the kernel raises DCP_DEVERR_TIMEOUT, stops all roles,
// drains what it issued and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "dcp_internal.cuh"
#include "dcp_tc_ptx.cuh"

namespace dcp {
namespace {

constexpr int kRows = 128;                 // query rows of a block (MMA M)
constexpr int kD = 128;                    // head dim (K and V)
constexpr int kTile = 64;                  // tokens per tile (MMA N of S, K of P.V)
constexpr int kStages = 4;
constexpr int kChunkBytes = kTile * 128;   // 64 rows x 64 bf16 (one 128-byte-swizzled box column)
constexpr int kKBytes = 2 * kChunkBytes;   // K rows of a tile: dims 0-63 | 64-127
constexpr int kStageBytes = 2 * kKBytes;   // K then V
constexpr int kPBytes = kRows * 128;       // 128 rows x 64 tokens bf16 (one term)

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr float kLoFraction = 1.0f / 32.0f;  // tile share of the row sum above which P_lo . V is issued

// Barriers: shared ones, then seven per block.
constexpr int BQ_EMPTY = 0, BDRAIN = 1, BKV_FULL = 2, BKV_EMPTY = 2 + kStages, BBLK = 2 + 2 * kStages;
constexpr int B_QF = 0, B_SF = 1, B_SE = 2, B_PF = 3, B_PE = 4, B_V0 = 5 /* 2, by tile parity */, kBlkBars = 7;

template <int NB>
struct TcCfg {
  static constexpr int kSoftmaxWarps = 4 * NB;
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 2);  // + copy warp + MMA warp
  static constexpr int kCopyWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kOffKv = 0;
  static constexpr int kOffP = kOffKv + kStages * kStageBytes;  // block b: hi at kOffP + 2b kPBytes, lo after it
  static constexpr int kNumBars = BBLK + kBlkBars * NB;
  static constexpr int kOffBar = kOffP + 2 * NB * kPBytes;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;         // TMEM slot, abort flag, per block: 4 lo flags + 2 x 4 votes
  static constexpr int kSmemUsed = kOffMisc + 16 + NB * 48;
  static constexpr int kSmemBytes = kSmemUsed + 1024;              // slack to align the base to 1024
  // TMEM: O of block b at 128 b, S at 128 NB + 64 b, Q at 192 NB + 64 b
  static constexpr uint32_t kTmemCols = 256 * NB;
  __host__ __device__ static constexpr uint32_t col_o(int b) { return 128u * b; }
  __host__ __device__ static constexpr uint32_t col_s(int b) { return 128u * NB + 64u * b; }
  __host__ __device__ static constexpr uint32_t col_q(int b) { return 192u * NB + 64u * b; }
};

struct TcParams {
  CUtensorMap tm_k[kMaxShards];
  CUtensorMap tm_v[kMaxShards];
  ShardSet sh;
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  const char* ws;
  WsLayout L;
  float* o_parts;
  float* lses;
  int32_t* err;
  int B;      // row groups per shard: sequences x token groups
  int qlen;   // query tokens per sequence
  int G;      // token groups per sequence
  int tpr;    // query tokens per lane (NB * 128 / g)
  int g;      // query heads per KV head
  int Hq, Hkv, Bs;
  int box;    // rows of a copy box: min(block_size, 64)
  int gang;   // CTAs that run the same items, one token group each
  int n_gangs;
  float sl2;  // scale * log2(e)
};

// Geometry of one work item for member m of the gang (token group m of the
// item's gang of lanes), derived identically by every role.
struct ItemGeom {
  int lane, shard, b, tg, kvh, t0, t1, out_row, lo, hi, start;
};
__device__ __forceinline__ ItemGeom item_geom(const TcParams& p, int k, int m) {
  const ItemRec it = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k];
  const int lane = it.lane + m * p.Hkv;
  const LaneRec ln = reinterpret_cast<const LaneRec*>(p.ws + p.L.lanes_off)[lane];
  ItemGeom g;
  g.lane = lane;
  const int u = lane / p.Hkv;
  g.kvh = lane - u * p.Hkv;
  g.shard = u / p.B;
  const int rg = u - g.shard * p.B;
  g.b = rg / p.G;
  g.tg = rg - g.b * p.G;
  g.t0 = it.t0;
  g.t1 = it.t1;
  // a split range's pieces: this lane's rows, one per item of the gang
  g.out_row = it.out_row >= 0 ? ln.tmp_begin + (k - ln.item_begin) : -1;
  g.lo = ln.lo;
  g.hi = ln.hi;
  g.start = ln.start;
  return g;
}

template <int NB>
__global__ void __launch_bounds__(TcCfg<NB>::kThreads, 1) gqa_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<NB>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = saddr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  auto bbar = [&](int blk, int i) { return sbase + C::kOffBar + 8u * (BBLK + kBlkBars * blk + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  // per block: lo flags [4] (read by the MMA warp), then votes [2][4]
  auto lo_flags = [&](int blk) { return reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16 + 48 * blk); };

  if (threadIdx.x == 0) {
    bar_init(bar(BQ_EMPTY), 1);
    bar_init(bar(BDRAIN), 1);
    for (int s = 0; s < kStages; ++s) {
      bar_init(bar(BKV_FULL + s), 1);
      bar_init(bar(BKV_EMPTY + s), 1);
    }
    for (int blk = 0; blk < NB; ++blk) {
      bar_init(bbar(blk, B_QF), kRows);  // every softmax thread of the block wrote its query row
      bar_init(bbar(blk, B_SF), 1);
      bar_init(bbar(blk, B_SE), kRows);
      bar_init(bbar(blk, B_PF), kRows);
      bar_init(bbar(blk, B_PE), 1);
      bar_init(bbar(blk, B_V0), 4);      // one arrival per softmax warp of the block
      bar_init(bbar(blk, B_V0 + 1), 4);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == C::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(saddr(tmem_slot)),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // the plan's work runs belong to gangs of p.gang CTAs; member m of a gang
  // takes token group m of every item (CTAs past the last gang idle)
  const int* cta_begin = reinterpret_cast<const int*>(p.ws + p.L.cta_off);
  const int gang_id = blockIdx.x / p.gang, member = blockIdx.x - gang_id * p.gang;
  const int k_begin = gang_id < p.n_gangs ? cta_begin[gang_id] : 0;
  const int k_end = gang_id < p.n_gangs ? cta_begin[gang_id + 1] : 0;
  const int pieces = kTile / p.box;  // copy boxes per tile (1, 2 or 4)

  if (warp == C::kCopyWarp) {
    // ------------------------------------------------------------ copy
    // Lane i < pieces looks up the block of piece i of the tile; lane 0
    // issues the boxes (K and V, two 64-column halves each).
    uint32_t fills = 0;
    bool stop = false;
    for (int k = k_begin; k < k_end && !stop; ++k) {
      const ItemGeom g = item_geom(p, k, member);
      const int32_t* table = p.sh.table[g.shard] + (size_t)g.b * p.sh.max_blocks[g.shard];
      const int local_hi = g.hi - g.start;
      for (int j = 0; j < g.t1 - g.t0; ++j) {
        const int lp0 = (g.lo - g.start) + (g.t0 + j) * kTile;  // local position of the tile's first token
        int row = -p.box;  // out of range: the box reads zeros
        if (lane < pieces) {
          const int lp = lp0 + lane * p.box;
          if (lp < local_hi) {  // a piece with tokens of the range
            const int lb = lp / p.Bs, off = lp - lb * p.Bs;
            if (lb >= p.sh.max_blocks[g.shard]) {
              raise_flag(p.err, DCP_DEVERR_TABLE_RANGE);
            } else {
              const int phys = table[lb];
              if (phys < 0 || phys >= p.sh.nblk[g.shard]) {
                raise_flag(p.err, DCP_DEVERR_BLOCK_RANGE);
              } else {
                row = (phys * p.Hkv + g.kvh) * p.Bs + off;
              }
            }
          }
        }
        int rows[4];  // the pieces' first pool rows, gathered by the whole warp
#pragma unroll
        for (int i = 0; i < 4; ++i) rows[i] = __shfl_sync(0xffffffffu, row, i);
        bool ok = true;
        if (lane == 0) {
          const uint32_t s = fills % kStages, use = fills / kStages;
          if (use > 0 && !wait_bar(bar(BKV_EMPTY + s), (use - 1) & 1u, abort_flag, p.err)) ok = false;
        }
        if (lane == 0 && ok) {
          const uint32_t s = fills % kStages;
          const uint32_t st = sbase + C::kOffKv + s * kStageBytes;
          bar_arrive_tx(bar(BKV_FULL + s), kStageBytes);  // pieces x box rows x (2 + 2) x 128 B
          for (int i = 0; i < pieces; ++i) {
            const uint32_t dst = st + i * p.box * 128;
            tma_load(dst, &p.tm_k[g.shard], 0, rows[i], bar(BKV_FULL + s));
            tma_load(dst + kChunkBytes, &p.tm_k[g.shard], 64, rows[i], bar(BKV_FULL + s));
            tma_load(dst + kKBytes, &p.tm_v[g.shard], 0, rows[i], bar(BKV_FULL + s));
            tma_load(dst + kKBytes + kChunkBytes, &p.tm_v[g.shard], 64, rows[i], bar(BKV_FULL + s));
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) { stop = true; break; }
        ++fills;
      }
    }
    if (lane == 0 && *abort_flag) {  // copies in flight must land before the CTA may exit
      const uint32_t f0 = fills > (uint32_t)kStages ? fills - kStages : 0;
      for (uint32_t f = f0; f < fills; ++f) drain_bar(bar(BKV_FULL + f % kStages), (f / kStages) & 1u);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // Per block: the score MMA of its next tile and the P.V of its oldest
    // tile whose P is ready go out as soon as their inputs are. A K/V stage
    // is released once every block's P.V of the tile has been issued.
    const uint32_t id_s = idesc(kRows, kTile, 0);
    const uint32_t id_pv = idesc(kRows, kD, 1);
    auto n_tiles = [&](int k) {
      const ItemRec it = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off)[k];
      return it.t1 - it.t0;
    };
    int ks[NB], js[NB], nts[NB], kp[NB], jp[NB], ntp[NB];
    uint32_t gs[NB], gp[NB];
    const int nt0 = k_begin < k_end ? n_tiles(k_begin) : 0;
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
      ks[blk] = kp[blk] = k_begin;
      js[blk] = jp[blk] = 0;
      nts[blk] = ntp[blk] = nt0;
      gs[blk] = gp[blk] = 0;
    }
    uint32_t q_loads = 0, released = 0;  // items whose queries were taken; tiles whose stage was released
    bool q_ready = false;
    uint32_t idle = 0;
    auto pv_left = [&]() {
      bool left = false;
#pragma unroll
      for (int blk = 0; blk < NB; ++blk) left |= kp[blk] < k_end;
      return left;
    };
    while (pv_left()) {
      bool progressed = false;
      // queries of the next item (all blocks)
      if (!q_ready && (int)q_loads < k_end - k_begin) {
        bool all = true;
#pragma unroll
        for (int blk = 0; blk < NB; ++blk) all = all && bar_test_warp(bbar(blk, B_QF), q_loads & 1u);
        if (all) {
          q_ready = true;
          tc_fence_after();
        }
      }
#pragma unroll
      for (int blk = 0; blk < NB; ++blk) {
        // scores of this block's next tile (the item whose queries are loaded)
        if (q_ready && ks[blk] < k_end && ks[blk] - k_begin == (int)q_loads) {
          const uint32_t g = gs[blk], s = g % kStages;
          if (bar_test_warp(bar(BKV_FULL + s), (g / kStages) & 1u) &&
              (g == 0 || bar_test_warp(bbar(blk, B_SE), (g - 1) & 1u))) {
            tc_fence_after();
            const uint64_t kd = sdesc(sbase + C::kOffKv + s * kStageBytes, 0);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ts(tmem + C::col_s(blk), tmem + C::col_q(blk) + 8 * kk,
                     kd + (uint64_t)((((kk >> 2) * kChunkBytes) + 32 * (kk & 3)) >> 4), id_s, kk > 0);
            mma_commit(bbar(blk, B_SF));
            if (++js[blk] == nts[blk]) {
              ++ks[blk];
              js[blk] = 0;
              nts[blk] = ks[blk] < k_end ? n_tiles(ks[blk]) : 0;
            }
            ++gs[blk];
            progressed = true;
          }
        }
        // P.V of this block's oldest tile whose P is ready
        if (gp[blk] < gs[blk] && bar_test_warp(bbar(blk, B_PF), gp[blk] & 1u)) {
          tc_fence_after();
          const uint32_t s = gp[blk] % kStages;
          const uint64_t vd = sdesc(sbase + C::kOffKv + s * kStageBytes + kKBytes, kChunkBytes);
          const uint64_t pd = sdesc(sbase + C::kOffP + 2 * blk * kPBytes, 0);
          volatile int* lf = lo_flags(blk);
          const int terms = (lf[0] | lf[1] | lf[2] | lf[3]) ? 2 : 1;
#pragma unroll
          for (int term = 0; term < 2; ++term) {
            if (term >= terms) break;
#pragma unroll
            for (int kt = 0; kt < kTile / 16; ++kt)
              mma_ss(tmem + C::col_o(blk), pd + (uint64_t)((term * kPBytes + 32 * kt) >> 4),
                     vd + (uint64_t)((2048 * kt) >> 4), id_pv, (jp[blk] == 0 && term == 0 && kt == 0) ? 0 : 1);
          }
          mma_commit(bbar(blk, B_PE));
          if (++jp[blk] == ntp[blk]) {
            ++kp[blk];
            jp[blk] = 0;
            ntp[blk] = kp[blk] < k_end ? n_tiles(kp[blk]) : 0;
          }
          ++gp[blk];
          progressed = true;
        }
      }
      // a stage is free once every block's P.V of its tile was issued
      {
        uint32_t gmin = gp[0];
#pragma unroll
        for (int blk = 1; blk < NB; ++blk) gmin = gp[blk] < gmin ? gp[blk] : gmin;
        while (released < gmin) {
          mma_commit(bar(BKV_EMPTY + released % kStages));
          ++released;
        }
      }
      // the queries of an item may be replaced once every block issued its last score MMA
      if (q_ready) {
        bool all = true;
#pragma unroll
        for (int blk = 0; blk < NB; ++blk) all = all && (ks[blk] - k_begin > (int)q_loads);
        if (all) {
          mma_commit(bar(BQ_EMPTY));
          ++q_loads;
          q_ready = false;
        }
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
    mma_commit(bar(BDRAIN));  // all issued MMAs complete before TMEM may be freed
    drain_bar(bar(BDRAIN), 0);
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int blk = warp >> 2;                  // the block this warp serves
    const int wq = warp & 3;                    // its TMEM lane quarter
    const int r = wq * 32 + lane;               // row of the block = TMEM lane
    const int rl = blk * kRows + r;             // row of the lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t col_o = C::col_o(blk), col_s = C::col_s(blk), col_q = C::col_q(blk);
    const uint32_t poff = sbase + C::kOffP + 2 * blk * kPBytes;
    volatile int* lf = lo_flags(blk);
    const int js_row = rl / p.g, h = rl - js_row * p.g;  // token slot and head of the row
    // A negative scale is taken as q -> -q (exact in bf16) with |scale|, so
    // that the row max of the scaled scores is always |sl2| x the raw max.
    const uint32_t qflip = p.sl2 < 0.f ? 0x80008000u : 0u;
    const float sl2 = fabsf(p.sl2);
    uint32_t gt = 0;
    int n_items = 0;
    bool ok = true;
    for (int k = k_begin; k < k_end && ok; ++k) {
      const ItemGeom g = item_geom(p, k, member);
      const int nt = g.t1 - g.t0;
      const int jt = g.tg * p.tpr + js_row;  // this row's query token
      const bool active = jt < p.qlen;
      // a warp whose rows all lie past the last query token (a partial token
      // group) keeps the per-tile barrier protocol but does no softmax: the
      // P.V rows it would feed belong to rows whose outputs are not written.
      // (One block per CTA only: with two, the extra live range costs spills.)
      const bool idle = NB == 1 && __all_sync(0xffffffffu, !active);
      // causal limit of the row's token (global positions); inactive rows attend nothing
      const int hi_r = active ? min(g.hi, p.seq_lens[g.b] - (p.qlen - 1 - jt)) : g.lo;
      const size_t qrow = ((size_t)g.b * p.qlen + (active ? jt : 0)) * p.Hq + (size_t)g.kvh * p.g + h;
      // the row's query into TMEM (after the previous item's score MMAs)
      if (n_items > 0 && !wait_warp(bar(BQ_EMPTY), (n_items - 1) & 1, abort_flag, p.err)) break;
      tc_fence_after();
      {
        const uint4* qr = reinterpret_cast<const uint4*>(p.q + qrow * kD);
        uint32_t qv[32];
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = active ? qr[8 * c + i] : make_uint4(0u, 0u, 0u, 0u);
            qv[4 * i] = v.x ^ qflip;
            qv[4 * i + 1] = v.y ^ qflip;
            qv[4 * i + 2] = v.z ^ qflip;
            qv[4 * i + 3] = v.w ^ qflip;
          }
          tmem_st32(tmem + lane_off + col_q + 32 * c, qv);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      bar_arrive(bbar(blk, B_QF));
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nt; ++j) {
        const uint32_t gi = gt + j, s = gi % kStages;
        const int tstart = g.lo + kTile * (g.t0 + j);  // global position of the tile's first token
        const int n_tile = min(kTile, g.hi - tstart);  // tokens of the range in the tile
        // inactive rows (past the last query token) take the full-tile path on
        // scores nobody reads, so that a warp mixing them with active rows does
        // not split into two paths; their O rows are never written or read
        const int n_valid = active ? max(0, min(n_tile, hi_r - tstart)) : kTile;
        // 1. scores of the tile
        if (!wait_warp(bbar(blk, B_SF), gi & 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64];
        if (!idle) {
          __syncwarp();
          tmem_ld32(tmem + lane_off + col_s, sv);
          tmem_ld32(tmem + lane_off + col_s + 32, sv + 32);
          tmem_wait_ld();
        }
        tc_fence_before();
        bar_arrive(bbar(blk, B_SE));
        // 2. online softmax over the tile's tokens (log2 units), causal per row.
        //    The scale is applied inside the exponent (one FMA per score):
        //    the row max of the scaled scores is sl2 times the raw max.
        float sc[64];
        float lsum = 0.f, alpha = 1.f;
        bool rescale = false;
        if (!idle) {
        float mx;
        if (n_valid == kTile) {
#pragma unroll
          for (int i = 0; i < 64; ++i) sc[i] = __uint_as_float(sv[i]);
          // a tree of three-input maxima: 64 -> 22 -> 8 -> 3 -> 1
          float t22[22], u8[8];
#pragma unroll
          for (int i = 0; i < 21; ++i) t22[i] = max3f(sc[3 * i], sc[3 * i + 1], sc[3 * i + 2]);
          t22[21] = sc[63];
#pragma unroll
          for (int i = 0; i < 7; ++i) u8[i] = max3f(t22[3 * i], t22[3 * i + 1], t22[3 * i + 2]);
          u8[7] = t22[21];
          mx = max3f(max3f(u8[0], u8[1], u8[2]), max3f(u8[3], u8[4], u8[5]), fmaxf(u8[6], u8[7]));
          mx *= sl2;
        } else {
          // a partial tile (the last of a range, or cut by the row's token):
          // masked scores become -inf after the scaling
          mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            sc[i] = i < n_valid ? __uint_as_float(sv[i]) : 0.f;
            mx = fmaxf(mx, i < n_valid ? sc[i] * sl2 : -INFINITY);
          }
        }
        float m_new = m_run;
        if (m_run == -INFINITY) {
          m_new = mx;
        } else if (mx > m_run + kRescaleThreshold) {
          m_new = mx;
          alpha = exp2f(m_run - m_new);
          rescale = true;
        }
        const float ref = m_new == -INFINITY ? 0.f : m_new;
        {
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
          if (n_valid == kTile) {
            // scale and shift two scores per instruction; row sum in pairs
            const unsigned long long s2 = f2pack(sl2, sl2), r2 = f2pack(-ref, -ref);
            unsigned long long a0 = f2pack(0.f, 0.f), a1 = a0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float x0, x1;
              f2unpack(ffma2(f2pack(sc[2 * i], sc[2 * i + 1]), s2, r2), x0, x1);
              sc[2 * i] = ex2_ftz(x0);
              sc[2 * i + 1] = ex2_ftz(x1);
              if (i & 1)
                a1 = fadd2(a1, f2pack(sc[2 * i], sc[2 * i + 1]));
              else
                a0 = fadd2(a0, f2pack(sc[2 * i], sc[2 * i + 1]));
            }
            float y0, y1;
            f2unpack(fadd2(a0, a1), y0, y1);
            ls[0] = y0;
            ls[1] = y1;
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              sc[i] = i < n_valid ? ex2_ftz(fmaf(sc[i], sl2, -ref)) : 0.f;
              ls[i & 3] += sc[i];
            }
          }
          lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
        }
        l_run = l_run * alpha + lsum;
        m_run = m_new;
        }  // !idle
        // The residual P_lo matters only where this tile carries more than
        // kLoFraction of some row's weight; the block's four softmax warps vote
        // (its P.V covers all 128 rows, so the residual is formed for all or none).
        bool any_lo;
        {
          const bool warp_lo = __any_sync(0xffffffffu, !idle && active && lsum > kLoFraction * l_run);
          volatile int* vote = lf + 4 + 4 * (gi & 1u);  // double-buffered by tile parity
          if (lane == 0) {
            vote[wq] = warp_lo ? 1 : 0;
            bar_arrive(bbar(blk, B_V0 + (gi & 1u)));
          }
          if (!wait_warp(bbar(blk, B_V0 + (gi & 1u)), (gi >> 1) & 1u, abort_flag, p.err)) { ok = false; break; }
          any_lo = (vote[0] | vote[1] | vote[2] | vote[3]) != 0;
        }
        // 3. the P buffer and O are free once the previous tile's P.V has finished
        if (gi >= 1 && !wait_warp(bbar(blk, B_PE), (gi - 1) & 1u, abort_flag, p.err)) { ok = false; break; }
        if (!idle) {
          const uint32_t hrow = poff + r * 128;
          const uint32_t lrow = hrow + kPBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t hi4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) hi4[e] = pack_bf16(sc[8 * c + 2 * e], sc[8 * c + 2 * e + 1]);
            st_shared_v4(hrow + (((uint32_t)c ^ (uint32_t)(r & 7)) << 4), hi4[0], hi4[1], hi4[2], hi4[3]);
          }
          if (any_lo) {  // rare: the first tiles of a range, dominant tokens
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t lo4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) lo4[e] = residual_bf16(sc[8 * c + 2 * e], sc[8 * c + 2 * e + 1]);
              st_shared_v4(lrow + (((uint32_t)c ^ (uint32_t)(r & 7)) << 4), lo4[0], lo4[1], lo4[2], lo4[3]);
            }
          }
        }
        if (lane == 0) lf[wq] = any_lo ? 1 : 0;
        // 4. value rows past the range's last token may hold anything: zero
        //    them (block 0's warps; a block's P.V waits for its own P only,
        //    so every block's softmax zeroes them: the stores are idempotent)
        if (n_tile < kTile) {
          const int zrows = kTile - n_tile;
          const uint32_t vbase = sbase + C::kOffKv + s * kStageBytes + kKBytes;
          for (int e = r; e < zrows * 16; e += kRows) {  // 16 pieces of 16 bytes per row (two halves)
            const int row = n_tile + e / 16, c = (e >> 3) & 1, piece = e & 7;
            st_shared_v4(vbase + c * kChunkBytes + row * 128 + piece * 16, 0u, 0u, 0u, 0u);
          }
        }
        // 5. lazy rescale of O (warp-wide: TMEM access is per warp; the others multiply by 1)
        if (__any_sync(0xffffffffu, rescale)) {
          tc_fence_after();
          uint32_t ov[32];
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < kD / 32; ++c) {
            tmem_ld32(tmem + lane_off + col_o + 32 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tmem + lane_off + col_o + 32 * c, ov);
          }
          tmem_wait_st();
        }
        // 6. publish P to the MMA issuer
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        tc_fence_before();
        bar_arrive(bbar(blk, B_PF));
      }
      if (!ok) break;
      // epilogue: wait for the last P.V, then write O / l and the LSE of the row
      const uint32_t glast = gt + nt - 1;
      if (!wait_warp(bbar(blk, B_PE), glast & 1u, abort_flag, p.err)) break;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      float* out = nullptr;
      float* out_lse = nullptr;
      if (g.out_row >= 0) {
        const size_t row = (size_t)g.out_row * (NB * kRows) + rl;
        out = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_o_off) + row * kD;
        out_lse = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_lse_off) + row;
      } else if (active) {
        const size_t row = ((size_t)g.shard * (p.B / p.G) * p.qlen + (size_t)g.b * p.qlen + jt) * p.Hq +
                           (size_t)g.kvh * p.g + h;
        out = p.o_parts + row * kD;
        out_lse = p.lses + row;
      }
      uint32_t ov[32];
      __syncwarp();
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        tmem_ld32(tmem + lane_off + col_o + 32 * c, ov);
        tmem_wait_ld();
        if (out) {
          float4* o4 = reinterpret_cast<float4*>(out + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o4[i] = make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                                __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
        }
      }
      if (out_lse) *out_lse = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      tc_fence_before();
      gt += nt;
      ++n_items;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(C::kTmemCols));
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 2-D bf16 map over the rows of a GQA pool ([blocks x Hkv x block_size] rows
// of 128 columns); boxes of 64 columns (128 bytes, 128-byte swizzle) by
// box_rows rows; out-of-range rows read 0.
bool pool_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {kD, rows};
  cuuint64_t strides[1] = {kD * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Resident CTAs (one per SM), cached per device.
template <int NB>
int tc_ctas_cached() {
  using C = TcCfg<NB>;
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] > 0) return cache[dev];
  if (cudaFuncSetAttribute(gqa_tc_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return 0;
  int occ = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gqa_tc_kernel<NB>, C::kThreads, C::kSmemBytes) !=
          cudaSuccess ||
      occ <= 0)
    return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = occ * sms;
  return cache[dev];
}

// Blocks of 128 rows per lane for a step: 2 once it has 256 rows per KV head.
int blocks_for(const dcp_attn_desc& d, int qlen) {
  const int g = d.num_q_heads / d.num_kv_heads;
  return (qlen * g >= 2 * kRows && (2 * kRows) % g == 0) ? 2 : 1;
}

}  // namespace

bool gqa_tc_eligible(const dcp_attn_desc& d, int qlen) {
  if (d.kind != DCP_KIND_GQA || d.kv_dtype != DCP_KV_BF16) return false;
  if (d.head_dim_k != kD || d.head_dim_v != kD) return false;
  const int g = d.num_q_heads / d.num_kv_heads;
  if (g < 1 || kRows % g != 0) return false;
  if (!(d.block_size % kTile == 0 || kTile % d.block_size == 0)) return false;
  // at least 3/8 of a lane's 128 rows carry query tokens: the kernel's time
  // per lane hardly depends on how many rows are filled, and from there it
  // beats the mma.sync teams (GQA mid: 3 tokens x 16 heads)
  return qlen * g >= 3 * kRows / 8;
}

int gqa_tc_rows_tokens(const dcp_attn_desc& d, int qlen) {
  return blocks_for(d, qlen) * kRows / (d.num_q_heads / d.num_kv_heads);
}

int gqa_tc_ctas(const dcp_attn_desc& d, const DeviceInfo&, int qlen) {
  return blocks_for(d, qlen) == 2 ? tc_ctas_cached<2>() : tc_ctas_cached<1>();
}

// Gang size for a step with `token_groups` lanes per (shard, sequence, KV
// head): the largest divisor up to 8. A prefill chunk's token groups all
// stream the same context; a CTA running them one after the other re-read it
// from HBM once per group (256-token chunks: 12.6x the unique KV bytes), a
// gang of CTAs runs them side by side and L2 serves the repeats.
int gqa_tc_gang(int token_groups, int n_ctas) {
  for (int c = token_groups < 8 ? token_groups : 8; c > 1; --c)
    if (token_groups % c == 0 && c <= n_ctas) return c;
  return 1;
}

cudaError_t launch_gqa_tc(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                          float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas, int gang,
                          int32_t* err, cudaStream_t st) {
  const int nb = blocks_for(d, rs.qlen);
  if (n_ctas <= 0 || gang < 1 || n_ctas < gang || (nb == 2 ? tc_ctas_cached<2>() : tc_ctas_cached<1>()) <= 0)
    return cudaErrorNotSupported;
  static_assert(sizeof(TcParams) <= 32000, "kernel parameters");
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int box = d.block_size < kTile ? d.block_size : kTile;
  for (int i = 0; i < rs.N; ++i) {
    const uint64_t rows = (uint64_t)sh.nblk[i] * d.num_kv_heads * d.block_size;
    if (!pool_map(&p.tm_k[i], sh.k[i], rows, box) || !pool_map(&p.tm_v[i], sh.v[i], rows, box))
      return cudaErrorNotSupported;
  }
  p.sh = sh;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.seq_lens = rs.seq_lens;
  p.ws = static_cast<const char*>(ws);
  p.L = L;
  p.o_parts = o_parts;
  p.lses = lses;
  p.err = err;
  p.B = rs.B;
  p.qlen = rs.qlen;
  p.tpr = rs.tpr;
  p.G = (rs.qlen + rs.tpr - 1) / rs.tpr;
  p.g = d.num_q_heads / d.num_kv_heads;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.Bs = d.block_size;
  p.box = box;
  p.gang = gang;
  p.n_gangs = n_ctas / gang;
  p.sl2 = d.scale * kLog2e;
  if (nb == 2)
    gqa_tc_kernel<2><<<n_ctas, TcCfg<2>::kThreads, TcCfg<2>::kSmemBytes, st>>>(p);
  else
    gqa_tc_kernel<1><<<n_ctas, TcCfg<1>::kThreads, TcCfg<1>::kSmemBytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace dcp
