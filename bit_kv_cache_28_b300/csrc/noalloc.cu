// kv_attention_noalloc: kv_attention for callers that cannot allocate device
// memory.  The scratch that kv_attention takes as a caller-provided workspace
// (the bounded-wait error word and the per-split partial outputs) lives here in
// one fixed, file-scope device array instead.
//
// Who needs it: code that runs where cudaMalloc is unavailable or forbidden --
// inside a host callback or a custom allocator's own hooks, in a process whose
// memory pool is owned by another framework, or in a plug-in that is handed
// only the input and output buffers.  Such a caller passes Q, Kcur, Vcur, the
// cache, `out` and `lse` exactly as for kv_attention and nothing else.
#include <mutex>

#include "common.cuh"

namespace bitkv {
namespace {

// Every GPU that loads the library holds this array until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[KV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Device address of the array, per device, looked up once.  It stays valid for the
// life of the device's primary context: after cudaDeviceReset() the module is
// loaded again elsewhere and the kept address is stale.
void* g_scratch_dev[kMaxDevices];

// Device address of the scratch array on the current device.  In host code the
// array's name only stands in for the symbol; the address must come from the
// runtime, once per device, with that device current.
kv_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "kv_attention_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(KV_ERR_UNSUPPORTED, "kv_attention_noalloc: device %d beyond the %d supported", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return set_error(KV_ERR_CUDA, "kv_attention_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return KV_OK;
}

}  // namespace
}  // namespace bitkv

using namespace bitkv;

extern "C" kv_status kv_attention_noalloc(const void* Q, const void* Kcur, const void* Vcur, kv_dtype dtype, int n_q,
                                          int n_cur, int Hq, const kv_cache* cache, const kv_attn_opts* opts,
                                          void* out, float* lse, void* stream) {
    AbiRange nvtx_range("kv_attention_noalloc");
    if (!cache) return set_error(KV_ERR_INVALID_ARG, "cache is NULL");
    if (n_q <= 0 || n_cur < 0 || Hq <= 0) return set_error(KV_ERR_INVALID_ARG, "bad sizes n_q=%d n_cur=%d Hq=%d", n_q, n_cur, Hq);
    kv_attn_opts o = opts ? *opts : kv_attn_opts{0.0f, KV_JENSEN_OFF, 0, 0, 0, KV_PATH_AUTO};
    const size_t cap = KV_NOALLOC_SCRATCH_BYTES;
    size_t need = kv_attention_workspace(cache, dtype, n_q, n_cur, Hq, &o);
    if (need > cap && o.num_splits == 0) {
        // automatic split count: take the largest count whose partials fit
        int32_t path = 0, splits = 1;
        kv_status s = kv_attention_plan(cache, dtype, n_q, n_cur, Hq, &o, &path, &splits);
        if (s != KV_OK) return s;
        for (int sp = splits - 1; sp >= 1 && need > cap; --sp) {
            o.num_splits = sp;
            need = kv_attention_workspace(cache, dtype, n_q, n_cur, Hq, &o);
        }
    }
    if (need > cap)
        return set_error(KV_ERR_WORKSPACE,
                         "kv_attention_noalloc: these sizes need %zu bytes of scratch; the fixed array holds %zu "
                         "(use fewer key-range splits or fewer query rows per call)",
                         need, cap);
    void* scratch = nullptr;
    kv_status s = scratch_address(&scratch);
    if (s != KV_OK) return s;
    return kv_attention(Q, Kcur, Vcur, dtype, n_q, n_cur, Hq, cache, &o, out, lse, scratch, cap, stream);
}

// The status words of the last no-alloc call sit at the start of the fixed array,
// where kv_attention put them; callers without a workspace read them here.
extern "C" kv_status kv_attention_noalloc_status(void* stream) {
    void* scratch = nullptr;
    const kv_status s = scratch_address(&scratch);
    if (s != KV_OK) return s;
    return read_status(scratch, static_cast<cudaStream_t>(stream));
}
