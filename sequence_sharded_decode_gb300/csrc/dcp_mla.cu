// MLA-absorbed partial decode attention (placeholder until the tcgen05 kernel lands).
#include "dcp_internal.cuh"

namespace dcp {

int mla_ctas(const dcp_attn_desc&, const DeviceInfo& di) { return di.sm_count; }

cudaError_t launch_mla(const dcp_attn_desc&, const void*, const ShardSet&, const RangeSpec&, float*, float*, void*,
                       const WsLayout&, int, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace dcp
