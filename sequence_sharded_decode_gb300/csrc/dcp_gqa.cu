// Partial decode attention, GQA form (step 2 of the method: each shard
// attends the one-token queries against its own KV slice only and emits a
// partial output and its LSE -- Qiita write-up "vLLMの-dcpが長文脈のKV
// キャッシュ重複を消して3倍速くする", section "トークンの区間でGPUに割り振る").
//
// One lane = (shard, sequence, KV head, group of up to 16 query heads). The
// group's 16 query rows are the M side of m16n8k16 bf16 tensor-core MMAs:
//   S[16 x 16 tokens] = Q[16 x D] . K^T  (D/16 MMAs per 8-token half)
//   O[16 x D]        += P[16 x 16] . V   (two MMAs per 8 output dims: P is
//                                          split into two bf16 terms)
// With 16 query heads per KV head this is 16 flop per KV byte, far below the
// tensor pipe's ridge; the kernel is bound by streaming K/V from HBM. Each
// warp owns a private cp.async pipeline of kStages 16-token tiles (K and V,
// one 16-byte chunk per lane per row, XOR-swizzled against ldmatrix bank
// conflicts) and its own online-softmax state over the tiles it takes
// (interleaved by warp); the warps' states are merged in shared memory at the
// end of each item. Scores are kept in log2 units (exp2 on the SFU).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "dcp_internal.cuh"
#include "dcp_tc_ptx.cuh"

namespace dcp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLoFraction = 1.0f / 32.0f;  // F8: tile share of a row's weight above which P_lo . V is issued

// F8: the cache holds FP8 E4M3 codes (1 byte per element) instead of bf16;
// a stage is then half as large. kMinCtas: with head dim 128 the 8-bit
// kernel (any team) and the bf16 kernel with teams of two are held to 168
// registers so that three CTAs (12 warps) share an SM, with 4 (8-bit) or 2
// (bf16) stages per warp: those kernels are bound by their per-tile
// instruction chains, and more resident warps hide its latencies. The bf16
// one-token kernel streams at the HBM rate with 2 CTAs and 3 stages.
__device__ __forceinline__ void mma16816_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_rn(float x0, float x1) {
  const __half2 h = __floats2half2_rn(x0, x1);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// hi = fp16(x), lo = fp16(x - hi), packed in pairs for an A fragment
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// four E4M3 codes (low byte first) -> two fp16 pairs: codes 0, 1 -> lo and
// 2, 3 -> hi (exact: every E4M3 value is an fp16 value)
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 2^x: F8 takes the SFU instruction with subnormal results flushed to zero
// (fewer instructions on its per-tile chain); the bf16 kernels keep exp2f
template <bool FTZ>
__device__ __forceinline__ float exp2_k(float x) {
  if constexpr (FTZ) {
    return ex2_ftz(x);
  } else {
    return exp2f(x);
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// bf16 pair -> fp16 pair
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  const __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D, bool F8 = false, int T = 1>
struct GqaCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kMinCtas = (D == 128 && (F8 || T == 2)) ? 3 : 1;
  static constexpr int kTile = 16;
  static constexpr int kElem = F8 ? 1 : 2;
  static constexpr int kStages = F8 ? (D == 128 ? 4 : 8) : (D == 128 ? (kMinCtas == 3 ? 2 : 3) : 4);
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunks = kRowBytes / 16;        // 16-byte chunks per K row
  static constexpr int kTileBytes = kTile * kRowBytes;  // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kSmem = kWarps * kWarpBytes + kWarps * kStages * 4;
  static_assert(16 * D * 4 + 32 * 4 <= kWarpBytes, "combine area must fit in a warp's stages");
};

struct GqaParams {
  const __nv_bfloat16* q;
  float v_scale;  // 8-bit cache: a value is v_scale * decode(code) (1 otherwise)
  ShardSet sh;
  const char* ws;
  WsLayout L;
  float* o_parts;
  float* lses;
  int32_t* err;
  const int32_t* seq_lens;
  int B;        // row groups per shard: sequences x token groups
  int Bseq;     // sequences
  int qlen;     // query tokens per sequence
  int ngroups;  // token groups per sequence: ceil(qlen / T)
  int Hq, Hkv, g, groups, Bs;
  int bs_log2;  // log2(Bs) when Bs is a power of two, else -1
  float sl2;    // scale * log2(e)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// hi = bf16(x), lo = bf16(x - hi), packed in pairs for an A fragment
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// T = warps per team = query tokens sharing each K/V tile (1, 2 or 4). The
// kWarps / T teams of a CTA take the item's tiles in turn; a team's warps
// copy each tile together into the team's ring (T * kStages stages) and then
// each warp runs its own query token's 16 head rows over it, so a tile is
// read once for T query tokens.
//
// F8 (8-bit cache: K as [blocks, Hkv, block_size, D] and V as
// [blocks, Hkv, D, block_size] E4M3 codes): the codes are widened to fp16 in
// registers (exactly) and the MMAs run on fp16 with the queries converted
// to fp16. The score MMA's k-slots (2t, 2t+1, 2t+8, 2t+9) of block kk take
// the head dims t*D/4 + 4kk .. +3 (the same order for q and K: the dot
// product is unchanged), so a lane reads its dims of a key row with 128-bit
// loads; its columns n take the tile's tokens 4*(n/2) + (n%2) (first half)
// and 4*(n/2) + 2 + (n%2) (second half), so that in the P.V product the
// tokens a lane holds, 4t .. 4t+3, are one 32-bit word of a transposed value
// row.
template <int D, int T, bool F8>
__global__ void __launch_bounds__(GqaCfg<D>::kThreads, (GqaCfg<D, F8, T>::kMinCtas))
    gqa_partial_kernel(const __grid_constant__ GqaParams p) {
  using C = GqaCfg<D, F8, T>;
  constexpr int kTeams = C::kWarps / T;
  constexpr int kS = T * C::kStages;  // stages of a team's ring
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / T, slot = warp - team * T;
  const int gr = lane >> 2, t4 = lane & 3;  // mma fragment row / column pair
  unsigned char* wbase = smem + warp * C::kWarpBytes;          // this warp's result area (after the item)
  unsigned char* tbase = smem + team * T * C::kWarpBytes;      // the team's ring
  int* vcount = reinterpret_cast<int*>(smem + C::kWarps * C::kWarpBytes) + team * kS;

  const LaneRec* lanes = reinterpret_cast<const LaneRec*>(p.ws + p.L.lanes_off);
  const ItemRec* items = reinterpret_cast<const ItemRec*>(p.ws + p.L.items_off);
  const int* cta_begin = reinterpret_cast<const int*>(p.ws + p.L.cta_off);
  float* tmp_o = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_o_off);
  float* tmp_lse = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.tmp_lse_off);

  const int k_begin = cta_begin[blockIdx.x], k_end = cta_begin[blockIdx.x + 1];
  const int lpu = p.Hkv * p.groups;
  const int rpl = p.L.rows_per_lane / T;  // head rows of one query token in a lane

  // the team's warps only: all of them have finished with what the barrier guards
  // (named barrier 1 + team, immediate ids so that the kernel reserves only those)
  auto team_sync = [&]() {
    if (T == 1) {
      __syncwarp();
    } else if (T == 4) {
      asm volatile("bar.sync 1, 128;\n" ::: "memory");
    } else if (team == 0) {
      asm volatile("bar.sync 1, 64;\n" ::: "memory");
    } else {
      asm volatile("bar.sync 2, 64;\n" ::: "memory");
    }
  };
  static_assert(T == 1 || T == 2 || T == 4, "team of 1, 2 or 4 warps");
  static_assert(C::kWarps == 4, "two teams of two or one team of four");

  for (int k = k_begin; k < k_end; ++k) {
    const ItemRec it = items[k];
    const LaneRec ln = lanes[it.lane];
    const int u = it.lane / lpu, j = it.lane - u * lpu;
    const int kvh = j / p.groups, hg = j - kvh * p.groups;
    const int shard = u / p.B, rg = u - shard * p.B;       // rg: row group = (sequence, token group)
    const int b = rg / p.ngroups, tg = rg - b * p.ngroups;
    const int jtok = tg * T + slot;                          // this warp's query token
    const bool active = jtok < p.qlen;
    const int qrow = b * p.qlen + (active ? jtok : 0);      // query row [sequence, token]
    // causal limit of this warp's token (global positions); inactive warps attend nothing
    const int hi_tok = p.qlen == 1 ? ln.hi : active ? min(ln.hi, p.seq_lens[b] - (p.qlen - 1 - jtok)) : ln.lo;
    const int head0 = kvh * p.g + hg * 16;
    const int nheads = min(16, p.g - hg * 16);

    const unsigned char* kpool = static_cast<const unsigned char*>(p.sh.k[shard]);
    const unsigned char* vpool = static_cast<const unsigned char*>(p.sh.v[shard]);
    const int32_t* table = p.sh.table[shard] + (size_t)b * p.sh.max_blocks[shard];
    const int max_blocks = p.sh.max_blocks[shard];
    const long long nblk = p.sh.nblk[shard];

    // Query fragments (A operand, rows = query heads of the group).
    uint32_t qa[D / 16][4];
    {
      const __nv_bfloat16* q0 = p.q + ((size_t)qrow * p.Hq + head0 + gr) * D;
      const __nv_bfloat16* q1 = q0 + 8 * D;
      const bool v0 = gr < nheads, v1 = gr + 8 < nheads;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        if constexpr (F8) {
          const int c = t4 * (D / 4) + 4 * kk;  // this lane's four dims of block kk
          qa[kk][0] = v0 ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(q0 + c)) : 0u;
          qa[kk][1] = v1 ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(q1 + c)) : 0u;
          qa[kk][2] = v0 ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(q0 + c + 2)) : 0u;
          qa[kk][3] = v1 ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(q1 + c + 2)) : 0u;
        } else {
          const int c = kk * 16 + 2 * t4;
          qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
          qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
          qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
          qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
        }
      }
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int n_total = it.t1 - it.t0;
    const int n_mine = n_total > team ? (n_total - team + kTeams - 1) / kTeams : 0;
    const int local0 = ln.lo - ln.start;  // local position of the lane's first token

    // F8: the block-table entries of the team's tiles, 32 tiles at a time
    // (lane j: tile i0 + j), each window loaded one window ahead, so that no
    // tile's copies wait for a table load (-1: past the table or the item).
    // Measured on GQA mid: 8-bit 0.266 -> 0.260 ms per step; the bf16
    // one-token kernel, at its register limit, lost 3.5 % with it.
    // block of a local position (F8: a shift when the block size is a power
    // of two; the bf16 kernels keep the division)
    auto block_of = [&](int lp) -> int { return (F8 && p.bs_log2 >= 0) ? lp >> p.bs_log2 : lp / p.Bs; };
    auto tbl_entry = [&](int i) -> int {
      const int lb = block_of(local0 + (it.t0 + team + i * kTeams) * C::kTile);
      return i < n_mine && lb < max_blocks ? table[lb] : -1;
    };
    int tw_cur = -1, tw_nxt = -1;
    if constexpr (F8) {
      tw_cur = tbl_entry(lane);
      tw_nxt = tbl_entry(32 + lane);
    }

    // Issue the team's loads of its i-th tile into stage i % kS; each warp
    // of the team copies every T-th 16-byte chunk. Called for i = 0, 1, 2,
    // ... in order, by every lane of the team's warps (F8: the table window).
    auto issue = [&](int i) {
      const int st = i % kS;
      const int tile = it.t0 + team + i * kTeams;
      const int g0 = ln.lo + tile * C::kTile;  // global position of the tile's first token
      int ntok = min(C::kTile, ln.hi - g0);
      const int lp = local0 + tile * C::kTile;
      const int lb = block_of(lp), slot_in_block = lp - lb * p.Bs;
      int phys = -1;
      if constexpr (F8) {
        if ((i & 31) == 0 && i > 0) {
          tw_cur = tw_nxt;
          tw_nxt = tbl_entry(i + 32 + lane);
        }
        phys = __shfl_sync(0xffffffffu, tw_cur, i & 31);
        if (lb >= max_blocks && lane == 0 && slot == 0) raise_flag(p.err, DCP_DEVERR_TABLE_RANGE);
      } else if (lb < max_blocks) {
        phys = table[lb];
      } else if (lane == 0 && slot == 0) {
        raise_flag(p.err, DCP_DEVERR_TABLE_RANGE);
      }
      if (phys < 0 || phys >= nblk) {
        if (lane == 0 && slot == 0 && lb < max_blocks) raise_flag(p.err, DCP_DEVERR_BLOCK_RANGE);
        ntok = 0;
        phys = 0;
      }
      if (lane == 0 && slot == 0) vcount[st] = ntok;
      const uint32_t kd = smem_u32(tbase + st * C::kStageBytes);
      const uint32_t vd = kd + C::kTileBytes;
      if constexpr (F8) {
        // K rows (16 tokens x D bytes, 16-byte chunks XOR-swizzled by row);
        // V as D transposed rows of the tile's 16 token bytes, zero past ntok
        const unsigned char* ks = kpool + (((size_t)phys * p.Hkv + kvh) * p.Bs + slot_in_block) * D;
        const unsigned char* vs = vpool + ((size_t)phys * p.Hkv + kvh) * D * p.Bs + slot_in_block;
#pragma unroll
        for (int c = slot * 32 + lane; c < D; c += 32 * T) {
          const int r = c / C::kChunks, ch = c - r * C::kChunks;
          const uint32_t so = r * C::kRowBytes + ((ch ^ (r & (C::kChunks - 1))) << 4);
          const int bytes = r < ntok ? 16 : 0;
          cp_async16(kd + so, ks + (bytes ? r * D + ch * 16 : 0), bytes);
          cp_async16(vd + c * 16, vs + (size_t)c * p.Bs, ntok);
        }
      } else {
        const size_t off = (((size_t)phys * p.Hkv + kvh) * p.Bs + slot_in_block) * D;
        const __nv_bfloat16* ks = reinterpret_cast<const __nv_bfloat16*>(kpool) + off;
        const __nv_bfloat16* vs = reinterpret_cast<const __nv_bfloat16*>(vpool) + off;
#pragma unroll
        for (int c = slot * 32 + lane; c < C::kTile * C::kChunks; c += 32 * T) {
          const int r = c / C::kChunks, ch = c - r * C::kChunks;
          const uint32_t so = r * C::kRowBytes + ((ch ^ (r & 7)) << 4);
          const int bytes = r < ntok ? 16 : 0;
          const int eo = bytes ? r * D + ch * 8 : 0;
          cp_async16(kd + so, ks + eo, bytes);
          cp_async16(vd + so, vs + eo, bytes);
        }
      }
    };

#pragma unroll
    for (int i = 0; i < kS - 1; ++i) {
      if (i < n_mine) issue(i);
      cp_async_commit();
    }

    for (int i = 0; i < n_mine; ++i) {
      if (T == 1) {
        if (i + kS - 1 < n_mine) issue(i + kS - 1);
        cp_async_commit();
        cp_async_wait<kS - 1>();
        __syncwarp();
      } else {
        // tile i has landed (this warp's part); after the barrier every
        // part is visible and no warp still reads the stage refilled next
        cp_async_wait<kS - 2>();
        team_sync();
        if (i + kS - 1 < n_mine) issue(i + kS - 1);
        cp_async_commit();
      }
      const int st = i % kS;
      const int g0 = ln.lo + (it.t0 + team + i * kTeams) * C::kTile;
      const int ntok = min(vcount[st], hi_tok - g0);  // this token's causal limit inside the tile
      const uint32_t kb = smem_u32(tbase + st * C::kStageBytes);
      const uint32_t vb = kb + C::kTileBytes;

      // S = Q K^T for the 16 tokens (two 8-token halves), even and odd
      // k-steps in separate accumulators so that four MMA chains overlap
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if constexpr (F8) {
        float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = 4 * (gr >> 1) + 2 * h + (gr & 1);  // the tile token of column gr of half h
          const uint32_t rb = kb + row * C::kRowBytes;
          uint32_t w[D / 16];  // word kk: this lane's dims t4*D/4 + 4kk .. +3
#pragma unroll
          for (int j = 0; j < D / 64; ++j) {
            const uint4 v = lds128(rb + (((t4 * (D / 64) + j) ^ (row & (C::kChunks - 1))) << 4));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(w[kk], b0, b1);
            mma16816_f16((kk & 1) ? s2[h] : s[h], qa[kk], b0, b1);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[h][e] += s2[h][e];
      } else {
        float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int mi = lane >> 3;
        const int r = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk += 2) {
          uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
          const int ch = 2 * kk + (mi & 1);
          ldsm_x4(kb + r * C::kRowBytes + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
          ldsm_x4(kb + r * C::kRowBytes + (((ch + 2) ^ (r & 7)) << 4), c0, c1, c2, c3);
          mma16816(s[0], qa[kk], b0, b1);
          mma16816(s[1], qa[kk], b2, b3);
          mma16816(s2[0], qa[kk + 1], c0, c1);
          mma16816(s2[1], qa[kk + 1], c2, c3);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[h][e] += s2[h][e];
      }
      // scale to log2 units and mask tokens past the range (F8: a full
      // tile, the common case, skips the mask)
      if (F8 && ntok >= C::kTile) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[h][e] *= p.sl2;
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = F8 ? 4 * t4 + 2 * h + (e & 1) : h * 8 + 2 * t4 + (e & 1);
            s[h][e] = tok < ntok ? s[h][e] * p.sl2 : -INFINITY;
          }
        }
      }
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      // reference maxima (a row with nothing seen yet keeps 0 to avoid inf - inf)
      const float r0 = n0 == -INFINITY ? 0.f : n0;
      const float r1 = n1 == -INFINITY ? 0.f : n1;
      const float a0 = exp2_k<F8>(m0 - r0), a1 = exp2_k<F8>(m1 - r1);
      m0 = n0;
      m1 = n1;
      float p_[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        p_[h][0] = exp2_k<F8>(s[h][0] - r0);
        p_[h][1] = exp2_k<F8>(s[h][1] - r0);
        p_[h][2] = exp2_k<F8>(s[h][2] - r1);
        p_[h][3] = exp2_k<F8>(s[h][3] - r1);
      }
      const float t0 = p_[0][0] + p_[0][1] + p_[1][0] + p_[1][1];
      const float t1 = p_[0][2] + p_[0][3] + p_[1][2] + p_[1][3];
      l0 = l0 * a0 + t0;
      l1 = l1 * a1 + t1;
      // once the running maxima settle, a0 = a1 = 1 exactly: skip the rescale
      if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          o[nd][0] *= a0;
          o[nd][1] *= a0;
          o[nd][2] *= a1;
          o[nd][3] *= a1;
        }
      }
      // P as the sum of two bf16 terms (hi + residual): the P.V product then
      // carries ~16 mantissa bits of P instead of bf16's 8, so the partial
      // of a short shard (few tokens, |O| ~ |v|) keeps fp32-level accuracy.
      uint32_t pa[4], pl[4];
      // F8 (P in fp16: the hi term alone keeps 11 bits): the residual P.V is
      // issued only for tiles that carry more than 1/32 of some row's running
      // weight (the first tiles of a lane, or a dominant token); elsewhere
      // dropping it changes O by at most 2^-11 x that share x max|v|. Each
      // lane's partial tile sums bound its rows' (the quad adds them up), so
      // judging per lane is conservative; the vote keeps the warp uniform.
      bool any_lo = true;
      if constexpr (F8) {
        any_lo = __any_sync(0xffffffffu, t0 > kLoFraction * l0 || t1 > kLoFraction * l1);
        if (any_lo) {
          split_f16(p_[0][0], p_[0][1], pa[0], pl[0]);
          split_f16(p_[0][2], p_[0][3], pa[1], pl[1]);
          split_f16(p_[1][0], p_[1][1], pa[2], pl[2]);
          split_f16(p_[1][2], p_[1][3], pa[3], pl[3]);
        } else {
          pa[0] = f16x2_rn(p_[0][0], p_[0][1]);
          pa[1] = f16x2_rn(p_[0][2], p_[0][3]);
          pa[2] = f16x2_rn(p_[1][0], p_[1][1]);
          pa[3] = f16x2_rn(p_[1][2], p_[1][3]);
        }
      } else {
        split_bf16(p_[0][0], p_[0][1], pa[0], pl[0]);
        split_bf16(p_[0][2], p_[0][3], pa[1], pl[1]);
        split_bf16(p_[1][0], p_[1][1], pa[2], pl[2]);
        split_bf16(p_[1][2], p_[1][3], pa[3], pl[3]);
      }
      // O += P V
      if constexpr (F8) {
        // a lane's tokens 4t4 .. 4t4+3 of value row (dim) 8nd + gr: one word.
        // The tile's 16-byte value rows are ldmatrix's 8 x 8 b16 matrices
        // (lane 4 gr + t4 receives word t4 of row gr), so one x4 load brings
        // the words of four consecutive nd (lane L addresses row 32 q + L)
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t w[4];
          ldsm_x4(vb + (32 * q + lane) * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(w[m], b0, b1);
            mma16816_f16(o[4 * q + m], pa, b0, b1);
            if (any_lo) mma16816_f16(o[4 * q + m], pl, b0, b1);
          }
        }
      } else {
        const int mi = lane >> 3;
        const int r = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
        for (int n2 = 0; n2 < D / 16; ++n2) {
          const int ch = 2 * n2 + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + r * C::kRowBytes + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
          mma16816(o[2 * n2], pa, b0, b1);
          mma16816(o[2 * n2 + 1], pa, b2, b3);
          mma16816(o[2 * n2], pl, b0, b1);
          mma16816(o[2 * n2 + 1], pl, b2, b3);
        }
      }
      if (T == 1) __syncwarp();
    }
    cp_async_wait<0>();

    // full row sums across the quad
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // this warp's (m, l, O) into its own part of the team's ring, once no
    // warp of the team reads the ring any more
    team_sync();
    float* wo = reinterpret_cast<float*>(wbase);
    float* wm = wo + 16 * D;
    float* wl = wm + 16;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int c = nd * 8 + 2 * t4;
      *reinterpret_cast<float2*>(wo + gr * D + c) = make_float2(o[nd][0], o[nd][1]);
      *reinterpret_cast<float2*>(wo + (gr + 8) * D + c) = make_float2(o[nd][2], o[nd][3]);
    }
    if (t4 == 0) {
      wm[gr] = m0;
      wm[gr + 8] = m1;
      wl[gr] = l0;
      wl[gr + 8] = l1;
    }
    __syncthreads();

    // merge the teams' states of every query token and write the lane's
    // partial: row R = (token slot js, head r) combines warps js, js + T, ...
    const int rows = T * nheads;
    float* out_o;  // row (js, r) of the lane: out_o[(js * js_rows + r) * D], out_l[js * js_rows + r]
    float* out_l;
    int js_rows;
    if (it.out_row >= 0) {
      out_l = tmp_lse + (size_t)it.out_row * p.L.rows_per_lane;
      out_o = tmp_o + (size_t)it.out_row * p.L.rows_per_lane * D;
      js_rows = rpl;
    } else {
      const size_t row0 = ((size_t)shard * p.Bseq * p.qlen + (size_t)b * p.qlen + tg * T) * p.Hq + head0;
      out_l = p.lses + row0;
      out_o = p.o_parts + row0 * D;
      js_rows = p.Hq;
    }
    for (int idx = threadIdx.x; idx < rows * D; idx += C::kThreads) {
      const int R = idx / D, c = idx - R * D;
      const int js = T == 1 ? 0 : R / nheads, r = R - js * nheads;
      if (T > 1 && tg * T + js >= p.qlen) continue;
      float M = -INFINITY;
#pragma unroll
      for (int tm = 0; tm < kTeams; ++tm)
        M = fmaxf(M, reinterpret_cast<const float*>(smem + (tm * T + js) * C::kWarpBytes)[16 * D + r]);
      float num = 0.f, den = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int tm = 0; tm < kTeams; ++tm) {
          const float* ws = reinterpret_cast<const float*>(smem + (tm * T + js) * C::kWarpBytes);
          const float mw = ws[16 * D + r];
          const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
          num += sc * ws[r * D + c];
          den += sc * ws[16 * D + 16 + r];
        }
      }
      const size_t row = (size_t)js * js_rows + r;
      out_o[row * D + c] = den > 0.f ? (F8 ? num / den * p.v_scale : num / den) : 0.f;
      if (c == 0) out_l[row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
    __syncthreads();
  }
}

// Resident CTAs per SM for the kernel, cached per device (the attribute is
// set once per device, before the first launch there).
template <int D, int T, bool F8>
int occupancy() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int occ = 0;
  using C = GqaCfg<D, F8, T>;
  if (cudaFuncSetAttribute(gqa_partial_kernel<D, T, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
      cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gqa_partial_kernel<D, T, F8>, C::kThreads, C::kSmem) !=
      cudaSuccess)
    return 0;
  if (dev < 64) cache[dev] = occ;
  return occ;
}

template <int D, bool F8>
int occupancy_for(int team) {
  return team == 4 ? occupancy<D, 4, F8>() : team == 2 ? occupancy<D, 2, F8>() : occupancy<D, 1, F8>();
}

template <int D, bool F8>
void launch_t(const GqaParams& p, int team, int n_ctas, cudaStream_t st) {
  using C4 = GqaCfg<D, F8, 4>;
  using C2 = GqaCfg<D, F8, 2>;
  using C1 = GqaCfg<D, F8, 1>;
  if (team == 4)
    gqa_partial_kernel<D, 4, F8><<<n_ctas, C4::kThreads, C4::kSmem, st>>>(p);
  else if (team == 2)
    gqa_partial_kernel<D, 2, F8><<<n_ctas, C2::kThreads, C2::kSmem, st>>>(p);
  else
    gqa_partial_kernel<D, 1, F8><<<n_ctas, C1::kThreads, C1::kSmem, st>>>(p);
}

}  // namespace

int gqa_team(int qlen) { return qlen >= 3 ? 4 : qlen; }

int gqa_ctas(const dcp_attn_desc& d, const DeviceInfo& di, int team) {
  const bool f8 = d.kv_dtype == DCP_KV_FP8_E4M3;
  const int occ = d.head_dim_k == 128 ? (f8 ? occupancy_for<128, true>(team) : occupancy_for<128, false>(team))
                                      : (f8 ? occupancy_for<64, true>(team) : occupancy_for<64, false>(team));
  return occ > 0 ? occ * di.sm_count : 0;
}

cudaError_t launch_gqa(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                       float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas, int32_t* err,
                       cudaStream_t st) {
  const int team = rs.tpr;
  if (team != 1 && team != 2 && team != 4) return cudaErrorInvalidValue;
  const bool f8 = d.kv_dtype == DCP_KV_FP8_E4M3;
  GqaParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.v_scale = f8 ? d.v_scale : 1.f;
  p.sh = sh;
  p.ws = static_cast<const char*>(ws);
  p.L = L;
  p.o_parts = o_parts;
  p.lses = lses;
  p.err = err;
  p.seq_lens = rs.seq_lens;
  p.B = rs.B;
  p.qlen = rs.qlen;
  p.ngroups = (rs.qlen + team - 1) / team;
  p.Bseq = rs.B / p.ngroups;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.g = d.num_q_heads / d.num_kv_heads;
  p.groups = (p.g + 15) / 16;
  p.bs_log2 = -1;
  for (int e2 = 0; e2 < 31; ++e2)
    if (d.block_size == (1 << e2)) p.bs_log2 = e2;
  p.Bs = d.block_size;
  p.sl2 = d.scale * (f8 ? d.k_scale : 1.f) * kLog2e;
  if (d.head_dim_k == 128) {
    if (f8) launch_t<128, true>(p, team, n_ctas, st);
    else launch_t<128, false>(p, team, n_ctas, st);
  } else {
    if (f8) launch_t<64, true>(p, team, n_ctas, st);
    else launch_t<64, false>(p, team, n_ctas, st);
  }
  return cudaGetLastError();
}

}  // namespace dcp
