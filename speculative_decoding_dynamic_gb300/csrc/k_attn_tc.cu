// Stage 5 dispatch. The scratch of eagle_tree_attention starts with the
// status word (256 bytes reserved).

#include "eagle_internal.cuh"
#include "eagle_ws.h"

namespace eagle {

cudaError_t launch_attention_simt(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                                  const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                                  int* status, cudaStream_t stream);

size_t attention_ws_bytes(const KvDims& /*kv*/, int /*T*/) { return 256; }

cudaError_t launch_attention(const KvDims& kv, int T, const void* q, const void* cache, int layer,
                             const int32_t* prefix_len, const uint32_t* mask, const int32_t* n_tree, void* out,
                             void* /*ws*/, size_t /*ws_bytes*/, int* status, cudaStream_t stream) {
    return launch_attention_simt(kv, T, q, cache, layer, prefix_len, mask, n_tree, out, status, stream);
}

}  // namespace eagle
