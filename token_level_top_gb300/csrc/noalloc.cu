// noalloc.cu -- moe_dispatch_static: the capacity-capped dispatch for callers
// that cannot allocate device memory.
//
// Who needs it: a caller that only ever receives its input and output
// buffers -- a plugin inside an inference engine that owns every allocation,
// a real-time loop whose rules forbid allocating after start-up, code that
// runs where it has no allocator of its own to draw a workspace from.  Such a
// caller cannot hand moe_dispatch a workspace.  This entry point keeps the
// dispatch's scratch (top-k ids, preference prefixes, chunk histograms and
// ranks, bases, control words) in one fixed device array of this file instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds MOE_STATIC_SCRATCH_BYTES of it until the process exits.  Host
// code cannot use the array's name as a device address (on the host it names
// a stand-in object), so the device address is looked up with
// cudaGetSymbolAddress, with the caller's device current, on the first call
// made in each CUDA context (each device, and again after a device reset
// recreates the context and reloads the library's module there), and cached
// for that context.  That first call may load the module, so it should come
// before any stream capture.  Every call shares the array and it keeps the previous
// call's contents; the only word that must start at zero (the device status
// word) is cleared at the start of each call.  Calls that overlap on the GPU
// (different streams, or different host threads, without ordering between
// them) race on the array.
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = MOE_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kStaticScratchBytes];

struct StaticLayout {
    int nchunks = 0;
    size_t status = 0, ctrl = 0, ids = 0, prefs = 0, crank = 0, hist = 0, base = 0, ppart = 0;
    size_t total = 0;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

StaticLayout static_layout(const moe_config_t& c)
{
    const size_t T = static_cast<size_t>(c.T), E = static_cast<size_t>(c.E);
    const size_t k = static_cast<size_t>(c.k);
    StaticLayout L;
    L.nchunks = static_cast<int>((T + kChunk - 1) / kChunk);
    const size_t nch = static_cast<size_t>(L.nchunks);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += up256(bytes > 0 ? bytes : 1);
        return o;
    };
    L.status = take(256);
    L.ctrl = take(CTRL_WORDS * 4);
    L.ids = take(T * k * 4);
    L.prefs = take(T * static_cast<size_t>(pref_stride(c.E)));
    L.crank = take(T * k * 4);
    L.hist = take(k * nch * E * 4);
    L.base = take(dispatch_base_bytes(T, k, nch, E));  // + the replay's fallback storage
    L.ppart = take(nch * E * 4);
    L.total = off;
    return L;
}

// Device address of the scratch array in the current context: looked up on
// the first call in each context and cached under the context's id.  A new
// context (another device, or the device reset) has its own copy of the
// module and of the array, at an address of its own.
moe_status_t scratch_address(char** out)
{
    static std::mutex mu;
    static std::map<unsigned long long, void*> addr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    const unsigned long long ctx = context_id();
    std::lock_guard<std::mutex> lock(mu);
    auto it = ctx ? addr.find(ctx) : addr.end();
    if (it != addr.end()) {
        *out = static_cast<char*>(it->second);
        return MOE_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    if (ctx) addr[ctx] = p;
    *out = static_cast<char*>(p);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_static(const moe_config_t* cfg, const float* scores,
                                            int32_t* assign, int32_t* slot, uint8_t* flags,
                                            int32_t* counts, int32_t* offsets, int32_t* perm,
                                            float* combine_w, int32_t* n_rerouted,
                                            int32_t* n_dropped, int32_t* status_out, void* stream)
{
    if (!cfg || cfg->flags != 0) return MOE_ERR_INVALID_ARG;
    if (cfg->T < 0 || cfg->E <= 0 || cfg->k <= 0 || cfg->k > cfg->E || cfg->capacity < 0)
        return MOE_ERR_INVALID_ARG;
    if (cfg->capacity == 0 && !(cfg->cf > 0.0 && cfg->cf <= 100.0)) return MOE_ERR_INVALID_ARG;
    if (cfg->E > 255 || cfg->k > 8) return MOE_ERR_UNSUPPORTED;
    // the per-token arrays may be NULL when there are no tokens
    if (!counts || !offsets || !n_rerouted || !n_dropped ||
        (cfg->T > 0 && (!scores || !assign || !slot || !flags || !perm || !combine_w)))
        return MOE_ERR_INVALID_ARG;
    const StaticLayout L = static_layout(*cfg);
    if (L.total > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;  // batch too large for the array
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cfg->T == 0) {
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * cfg->E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (cfg->E + 1), s) != cudaSuccess ||
            cudaMemsetAsync(n_rerouted, 0, sizeof(int32_t), s) != cudaSuccess ||
            cudaMemsetAsync(n_dropped, 0, sizeof(int32_t), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (status_out && cudaMemsetAsync(status_out, 0, sizeof(int32_t), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    char* base = nullptr;
    moe_status_t st = scratch_address(&base);
    if (st != MOE_OK) return st;
    int* status = reinterpret_cast<int*>(base + L.status);
    if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;

    RouteArgs a{};
    a.T = cfg->T;
    a.E = cfg->E;
    a.k = cfg->k;
    a.d = cfg->d_model;
    a.splits = 1;
    a.epad = 32;
    a.nchunks = L.nchunks;
    a.logits_in = scores;
    a.ids_ws = reinterpret_cast<int32_t*>(base + L.ids);
    a.prefs = reinterpret_cast<uint8_t*>(base + L.prefs);
    a.crank = reinterpret_cast<int32_t*>(base + L.crank);
    a.hist = reinterpret_cast<int32_t*>(base + L.hist);
    a.ppart = reinterpret_cast<float*>(base + L.ppart);
    a.status = status;
    if (launch_route(a, s) != cudaSuccess) return MOE_ERR_CUDA;

    DispatchArgs d{};
    d.T = cfg->T;
    d.E = cfg->E;
    d.k = cfg->k;
    d.nchunks = L.nchunks;
    d.C = moe_capacity(cfg->T, cfg->k, cfg->E, cfg->cf, cfg->capacity);
    d.scores = scores;
    d.ids = a.ids_ws;
    d.prefs = a.prefs;
    d.crank = a.crank;
    d.hist = a.hist;
    d.base = reinterpret_cast<int32_t*>(base + L.base);
    d.ctrl = reinterpret_cast<int32_t*>(base + L.ctrl);
    d.assign = assign;
    d.slot = slot;
    d.flags = flags;
    d.counts = counts;
    d.offsets = offsets;
    d.perm = perm;
    d.cw = combine_w;
    d.n_rerouted = n_rerouted;
    d.n_dropped = n_dropped;
    d.status = status;
    if (launch_dispatch(d, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (status_out &&
        cudaMemcpyAsync(status_out, status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
