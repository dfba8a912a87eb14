// noalloc.cu -- dec_attention_static: one layer's decode attention with its
// split scratch in a fixed, library-owned device array instead of memory the
// caller or the library allocates.
//
// Why: some callers cannot allocate device memory at the point where they run
// attention.  A serving process that sized its weights and KV cache to fill
// the GPU up front has no memory left to hand out per call, and a latency-bound
// loop cannot absorb cudaMalloc / cudaFree, which may synchronise the whole
// device.  This entry point performs no allocation of any kind: the split
// partials and the completion counters live in one file-scope __device__ array
// of a fixed size.  Like dec_attention it runs on the handle's stream and
// waits (bounded) for its result.
//
// Costs and rules for a user:
//   * every GPU that loads this library reserves the array (about 2 MiB) until
//     the process exits;
//   * all calls on a device share the array and it keeps the contents of the
//     last call: the counters are cleared at the start of every call, and two
//     calls whose work overlaps on the GPU (different streams, or several host
//     threads) race on it -- serialise them;
//   * the first call on each device resolves the array's device address
//     (cudaGetSymbolAddress, with that device current) and keeps it for the
//     life of the process; make that first call before any stream capture.  A
//     cudaDeviceReset invalidates the address together with every handle;
//   * shapes whose partials exceed the array are refused with
//     DEC_E_UNSUPPORTED, and the handle stays usable.
#include <mutex>

#include "graphdec.h"
#include "internal.h"

namespace {

// split partials first, then the completion counters
constexpr size_t STATIC_PART_FLOATS = (size_t)1 << 19;   // 2 MiB of fp32 partials
constexpr size_t STATIC_COUNTERS = 1024;
__device__ __align__(256) float g_attn_scratch[STATIC_PART_FLOATS + STATIC_COUNTERS];

constexpr int MAX_DEVICES = 64;
float* g_scratch_ptr[MAX_DEVICES];
std::mutex g_scratch_mu;

// the array's device address on `device` (host code cannot use the symbol
// itself: on the host it names a stand-in, not device memory)
cudaError_t scratch_on(int device, float** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (device < 0 || device >= MAX_DEVICES) return cudaErrorInvalidDevice;
    if (!g_scratch_ptr[device]) {
        int prev = 0;
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return e;
        if ((e = cudaSetDevice(device)) != cudaSuccess) return e;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        cudaSetDevice(prev);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[device] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[device];
    return cudaSuccess;
}

}  // namespace

extern "C" int dec_attention_static(dec_handle* h, int32_t layer, const float* qkv, const int32_t* pos, float* out) {
    int rc = gd::engine_gate(h);
    if (rc) return rc;
    size_t need_part = 0, need_ctr = 0;
    gd::engine_attention_scratch(h, &need_part, &need_ctr);
    if (need_part > STATIC_PART_FLOATS || need_ctr > STATIC_COUNTERS)
        return gd::engine_fail(h, DEC_E_UNSUPPORTED,   // refused before any device work: the handle stays usable
                               "dec_attention_static: this shape needs more split scratch than the fixed "
                               "2 MiB array holds (rows * n_heads * splits * (head_dim + 4) floats)");
    float* base = nullptr;
    cudaError_t e = scratch_on(gd::engine_device(h), &base);
    if (e != cudaSuccess) return gd::engine_fail(h, DEC_E_CUDA, "dec_attention_static: cudaGetSymbolAddress failed");
    unsigned* counters = reinterpret_cast<unsigned*>(base + STATIC_PART_FLOATS);
    void* stream = nullptr;
    if ((rc = dec_stream(h, &stream)) != DEC_OK) return rc;
    // the completion counters must start at zero (the array keeps the last call's contents)
    e = cudaMemsetAsync(counters, 0, need_ctr * sizeof(unsigned), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return gd::engine_fail(h, DEC_E_CUDA, "dec_attention_static: counter clear failed");
    return gd::engine_run_attention(h, layer, qkv, pos, out, base, counters);
}
