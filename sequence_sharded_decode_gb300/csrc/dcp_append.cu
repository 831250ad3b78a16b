// Per-step KV append into the owning shard's paged pool.
//
// Decoding proceeds one token at a time and every new token's K/V joins the
// cache ("Inference Systems Infrastructure Notes (7): DCP", sections 1 and 4);
// under sequence sharding it goes to the shard that owns its position. The
// owner of global position t is the last shard whose start is <= t (the
// contiguous ranges of the Qiita write-up "vLLMの-dcpが長文脈のKVキャッシュ
// 重複を消して3倍速くする", section "トークンの区間でGPUに割り振る"; the last
// shard is open-ended). The local position picks (logical block, slot) and
// the shard's block table gives the physical block. One warp per token copies
// the row(s) with 16-byte stores; bytes are moved unchanged.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr int kAppendThreads = 256;

struct AppendParams {
  ShardSet sh;
  const int32_t* starts;
  const int32_t* seq_ids;
  const int32_t* positions;
  const uint4* k_new;
  const uint4* v_new;
  int32_t* err;
  int N, B, T, Hkv, Bs;
  int k_vec;  // 16-byte vectors per token row of K (GQA: one head; MLA: the latent)
  int v_vec;
  int mla;
  int f8;     // 8-bit cache: values are stored transposed within a block
  int dv;     // head_dim_v (transposed values)
};

__global__ void __launch_bounds__(kAppendThreads) append_kernel(const __grid_constant__ AppendParams p) {
  const int lane = threadIdx.x & 31;
  const long long tok = (long long)blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5);
  if (tok >= p.T) return;
  const int b = p.seq_ids ? p.seq_ids[tok] : (int)tok;
  const int t = p.positions[tok];
  if (b < 0 || b >= p.B || t < 0) {
    if (lane == 0) raise_flag(p.err, DCP_DEVERR_POSITION);
    return;
  }
  const int32_t* st = p.starts + (size_t)b * p.N;
  int owner = -1;
  for (int i = 0; i < p.N; ++i)
    if (st[i] <= t) owner = i;
  if (owner < 0) {
    if (lane == 0) raise_flag(p.err, DCP_DEVERR_POSITION);
    return;
  }
  const int local = t - st[owner];
  const int lb = local / p.Bs, slot = local - lb * p.Bs;
  if (lb >= p.sh.max_blocks[owner]) {
    if (lane == 0) raise_flag(p.err, DCP_DEVERR_TABLE_RANGE);
    return;
  }
  const int phys = p.sh.table[owner][(size_t)b * p.sh.max_blocks[owner] + lb];
  if (phys < 0 || phys >= p.sh.nblk[owner]) {
    if (lane == 0) raise_flag(p.err, DCP_DEVERR_BLOCK_RANGE);
    return;
  }
  uint4* kp = static_cast<uint4*>(const_cast<void*>(p.sh.k[owner]));
  if (p.mla) {
    // pool [nblk, Bs, Dk]
    uint4* dst = kp + ((size_t)phys * p.Bs + slot) * p.k_vec;
    const uint4* src = p.k_new + (size_t)tok * p.k_vec;
    for (int c = lane; c < p.k_vec; c += 32) dst[c] = src[c];
    return;
  }
  // pools [nblk, Hkv, Bs, D]
  uint4* vp = static_cast<uint4*>(const_cast<void*>(p.sh.v[owner]));
  for (int c = lane; c < p.Hkv * p.k_vec; c += 32) {
    const int h = c / p.k_vec, e = c - h * p.k_vec;
    kp[(((size_t)phys * p.Hkv + h) * p.Bs + slot) * p.k_vec + e] = p.k_new[(size_t)tok * p.Hkv * p.k_vec + c];
  }
  if (p.f8) {  // value pool [nblk, Hkv, Dv, Bs]: byte d of head h goes to row d, column slot
    unsigned char* vb = static_cast<unsigned char*>(const_cast<void*>(p.sh.v[owner]));
    const unsigned char* src = reinterpret_cast<const unsigned char*>(p.v_new) + (size_t)tok * p.Hkv * p.dv;
    for (int c = lane; c < p.Hkv * p.dv; c += 32) {
      const int h = c / p.dv, d = c - h * p.dv;
      vb[(((size_t)phys * p.Hkv + h) * p.dv + d) * p.Bs + slot] = src[c];
    }
    return;
  }
  for (int c = lane; c < p.Hkv * p.v_vec; c += 32) {
    const int h = c / p.v_vec, e = c - h * p.v_vec;
    vp[(((size_t)phys * p.Hkv + h) * p.Bs + slot) * p.v_vec + e] = p.v_new[(size_t)tok * p.Hkv * p.v_vec + c];
  }
}

}  // namespace

cudaError_t launch_append(const dcp_attn_desc& d, const ShardSet& sh, int N, const int32_t* starts, int B,
                          const int32_t* seq_ids, const int32_t* positions, const void* k_new,
                          const void* v_new, int T, int32_t* err, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  AppendParams p;
  p.sh = sh;
  p.starts = starts;
  p.seq_ids = seq_ids;
  p.positions = positions;
  p.k_new = static_cast<const uint4*>(k_new);
  p.v_new = static_cast<const uint4*>(v_new);
  p.err = err;
  p.N = N;
  p.B = B;
  p.T = T;
  p.Hkv = d.num_kv_heads;
  p.Bs = d.block_size;
  const int elem = d.kv_dtype == DCP_KV_FP8_E4M3 ? 1 : 2;
  p.k_vec = d.head_dim_k * elem / 16;
  p.v_vec = d.head_dim_v * elem / 16;
  p.mla = d.kind == DCP_KIND_MLA;
  p.f8 = d.kv_dtype == DCP_KV_FP8_E4M3;
  p.dv = d.head_dim_v;
  const long long blocks = ((long long)T + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
  append_kernel<<<(unsigned)blocks, kAppendThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace dcp
