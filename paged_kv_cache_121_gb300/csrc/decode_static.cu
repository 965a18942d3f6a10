// pa_decode_static_scratch: paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: an engine
// whose device memory is reserved up front by another allocator (a call to
// cudaMalloc there would fail, or would bypass the engine's accounting), or a
// plugin interface that passes only the operation's inputs and outputs. For
// them this entry point runs the same decode as pa_decode, with the context
// split merged through a fixed scratch array that lives in the library itself
// (a file-scope device array, resident on every GPU that loads the library
// until the process exits). The caller still passes the inputs and outputs.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>

#include "../../include/pa.h"
#include "internal.h"

namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(PA_STATIC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

// The scratch itself. Host code must not pass this name to a kernel: on the
// host it is only a stand-in symbol, not a device address.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
pa_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" PA_API pa_status pa_decode_static_scratch(
    void *out, pa_dtype out_dtype, const void *query, pa_dtype q_dtype, const void *k_cache,
    const void *v_cache, pa_dtype kv_dtype, const int32_t *block_tables, const int32_t *context_lens,
    int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, int max_context_len, float scale, void *stream) {
    void *scratch = nullptr;
    const pa_status st = pa::scratch_address(&scratch);
    if (st != PA_OK) return st;
    pa::DecodeCall c;
    c.out = out;
    c.out_dtype = out_dtype;
    c.query = query;
    c.q_dtype = q_dtype;
    c.k_cache = k_cache;
    c.v_cache = v_cache;
    c.kv_dtype = kv_dtype;
    c.block_tables = block_tables;
    c.context_lens = context_lens;
    c.num_seqs = num_seqs;
    c.num_heads = num_heads;
    c.num_kv_heads = num_kv_heads;
    c.head_dim = head_dim;
    c.block_size = block_size;
    c.max_blocks_per_seq = max_blocks_per_seq;
    c.num_blocks = num_blocks;
    c.max_context_len = max_context_len;
    c.scale = scale;
    return static_cast<pa_status>(pa::decode_into_scratch(c, scratch, pa::kStaticScratchBytes, stream));
}
