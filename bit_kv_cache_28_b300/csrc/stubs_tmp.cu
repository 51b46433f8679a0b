#include "common.cuh"
namespace bitkv {
kv_status launch_codebook_fit(const void*, kv_dtype, int, const kv_cache*, int, const void*, int, float*, void*, cudaStream_t) { return set_error(KV_ERR_UNSUPPORTED, "codebook not built"); }
size_t codebook_ws_bytes(const kv_layout*, int) { return 0; }
kv_status launch_psac_basis(const void*, kv_dtype, int, const kv_cache*, float*, void*, cudaStream_t) { return set_error(KV_ERR_UNSUPPORTED, "psac not built"); }
size_t psac_ws_bytes(const kv_layout*) { return 0; }
}
