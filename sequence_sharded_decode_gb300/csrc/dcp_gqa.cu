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

#include <cmath>
#include <mutex>

#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct GqaCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTile = 16;
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = D / 8;                 // 16-byte chunks per row
  static constexpr int kTileBytes = kTile * kRowBytes;  // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kSmem = kWarps * kWarpBytes + kWarps * kStages * 4;
  static_assert(16 * D * 4 + 32 * 4 <= kWarpBytes, "combine area must fit in a warp's stages");
};

struct GqaParams {
  const __nv_bfloat16* q;
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
template <int D, int T>
__global__ void __launch_bounds__(GqaCfg<D>::kThreads) gqa_partial_kernel(const __grid_constant__ GqaParams p) {
  using C = GqaCfg<D>;
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

    const __nv_bfloat16* kpool = static_cast<const __nv_bfloat16*>(p.sh.k[shard]);
    const __nv_bfloat16* vpool = static_cast<const __nv_bfloat16*>(p.sh.v[shard]);
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
        const int c = kk * 16 + 2 * t4;
        qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
        qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
        qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
        qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
      }
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int n_total = it.t1 - it.t0;
    const int n_mine = n_total > team ? (n_total - team + kTeams - 1) / kTeams : 0;
    const int local0 = ln.lo - ln.start;  // local position of the lane's first token

    // Issue the team's loads of its i-th tile into stage i % kS; each warp
    // of the team copies every T-th 16-byte chunk.
    auto issue = [&](int i) {
      const int st = i % kS;
      const int tile = it.t0 + team + i * kTeams;
      const int g0 = ln.lo + tile * C::kTile;  // global position of the tile's first token
      int ntok = min(C::kTile, ln.hi - g0);
      const int lp = local0 + tile * C::kTile;
      const int lb = lp / p.Bs, slot_in_block = lp - lb * p.Bs;
      int phys = -1;
      if (lb < max_blocks) {
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
      const size_t off = (((size_t)phys * p.Hkv + kvh) * p.Bs + slot_in_block) * D;
      const __nv_bfloat16* ks = kpool + off;
      const __nv_bfloat16* vs = vpool + off;
      const uint32_t kd = smem_u32(tbase + st * C::kStageBytes);
      const uint32_t vd = kd + C::kTileBytes;
#pragma unroll
      for (int c = slot * 32 + lane; c < C::kTile * C::kChunks; c += 32 * T) {
        const int r = c / C::kChunks, ch = c - r * C::kChunks;
        const uint32_t so = r * C::kRowBytes + ((ch ^ (r & 7)) << 4);
        const int bytes = r < ntok ? 16 : 0;
        const int eo = bytes ? r * D + ch * 8 : 0;
        cp_async16(kd + so, ks + eo, bytes);
        cp_async16(vd + so, vs + eo, bytes);
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
      {
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
      // scale to log2 units and mask tokens past the range
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = h * 8 + 2 * t4 + (e & 1);
          s[h][e] = tok < ntok ? s[h][e] * p.sl2 : -INFINITY;
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
      const float a0 = exp2f(m0 - r0), a1 = exp2f(m1 - r1);
      m0 = n0;
      m1 = n1;
      float p_[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        p_[h][0] = exp2f(s[h][0] - r0);
        p_[h][1] = exp2f(s[h][1] - r0);
        p_[h][2] = exp2f(s[h][2] - r1);
        p_[h][3] = exp2f(s[h][3] - r1);
      }
      l0 = l0 * a0 + (p_[0][0] + p_[0][1] + p_[1][0] + p_[1][1]);
      l1 = l1 * a1 + (p_[0][2] + p_[0][3] + p_[1][2] + p_[1][3]);
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
      split_bf16(p_[0][0], p_[0][1], pa[0], pl[0]);
      split_bf16(p_[0][2], p_[0][3], pa[1], pl[1]);
      split_bf16(p_[1][0], p_[1][1], pa[2], pl[2]);
      split_bf16(p_[1][2], p_[1][3], pa[3], pl[3]);
      // O += P V
      {
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
      out_o[row * D + c] = den > 0.f ? num / den : 0.f;
      if (c == 0) out_l[row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
    __syncthreads();
  }
}

// Resident CTAs per SM for the kernel, cached per device (the attribute is
// set once per device, before the first launch there).
template <int D, int T>
int occupancy() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int occ = 0;
  if (cudaFuncSetAttribute(gqa_partial_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GqaCfg<D>::kSmem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gqa_partial_kernel<D, T>, GqaCfg<D>::kThreads,
                                                    GqaCfg<D>::kSmem) != cudaSuccess)
    return 0;
  if (dev < 64) cache[dev] = occ;
  return occ;
}

template <int D>
int occupancy_for(int team) {
  return team == 4 ? occupancy<D, 4>() : team == 2 ? occupancy<D, 2>() : occupancy<D, 1>();
}

template <int D, int T>
void launch_t(const GqaParams& p, int n_ctas, cudaStream_t st) {
  gqa_partial_kernel<D, T><<<n_ctas, GqaCfg<D>::kThreads, GqaCfg<D>::kSmem, st>>>(p);
}

}  // namespace

int gqa_team(int qlen) { return qlen >= 3 ? 4 : qlen; }

int gqa_ctas(const dcp_attn_desc& d, const DeviceInfo& di, int team) {
  const int occ = d.head_dim_k == 128 ? occupancy_for<128>(team) : occupancy_for<64>(team);
  return occ > 0 ? occ * di.sm_count : 0;
}

cudaError_t launch_gqa(const dcp_attn_desc& d, const void* q, const ShardSet& sh, const RangeSpec& rs,
                       float* o_parts, float* lses, void* ws, const WsLayout& L, int n_ctas, int32_t* err,
                       cudaStream_t st) {
  const int team = rs.tpr;
  if (team != 1 && team != 2 && team != 4) return cudaErrorInvalidValue;
  GqaParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
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
  p.Bs = d.block_size;
  p.sl2 = d.scale * kLog2e;
  if (d.head_dim_k == 128) {
    if (team == 4) launch_t<128, 4>(p, n_ctas, st);
    else if (team == 2) launch_t<128, 2>(p, n_ctas, st);
    else launch_t<128, 1>(p, n_ctas, st);
  } else {
    if (team == 4) launch_t<64, 4>(p, n_ctas, st);
    else if (team == 2) launch_t<64, 2>(p, n_ctas, st);
    else launch_t<64, 1>(p, n_ctas, st);
  }
  return cudaGetLastError();
}

}  // namespace dcp
