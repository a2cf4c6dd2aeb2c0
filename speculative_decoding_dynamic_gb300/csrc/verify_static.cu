// eagle_verify_static: stage 6 without a caller-provided workspace.
//
// Who needs this: some callers are not allowed to allocate device memory at
// all. Typical cases are a plugin inside an inference engine whose memory
// planner owns every byte of the GPU and refuses allocations after start-up,
// or a latency-critical decode loop that must never take the allocator's
// locks. Such a caller can still hand us its inputs and outputs, but it cannot
// give us the per-row scratch that eagle_verify keeps in its workspace.
//
// This entry point therefore keeps that scratch in one fixed device array of
// this file, sized for at most kMaxRows target rows (batch * (node_budget + 1))
// and kMaxSeqs sequences. The array exists once per GPU that loads the library
// and stays allocated until the process exits. Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
//
// The kernels are the ones eagle_verify launches; only the place of the
// scratch differs.

#include <nvtx3/nvToolsExt.h>
#include <mutex>

#include "../../include/eagle.h"
#include "eagle_ws.h"

namespace eagle {

namespace {

constexpr int kMaxRows = 4096;  // batch * T
constexpr int kMaxSeqs = 1024;  // batch

// Byte offsets inside the fixed scratch array.
constexpr size_t kOffStatus = 0;
constexpr size_t kOffTicket = 256;
constexpr size_t kOffRowMax = kOffTicket + kMaxSeqs * sizeof(int);
constexpr size_t kOffRowArg = kOffRowMax + kMaxRows * sizeof(float);
constexpr size_t kOffRowMass = kOffRowArg + kMaxRows * sizeof(int32_t);
constexpr size_t kOffPMass = kOffRowMass + kMaxRows * sizeof(uint64_t);
constexpr size_t kScratchBytes = kOffPMass + kMaxRows * sizeof(uint64_t);

static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device; the host-side symbol itself is not a device address).
cudaError_t scratch_address(unsigned char** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_verify_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace eagle

using namespace eagle;

extern "C" int eagle_verify_static(const eagle_tree_cfg* cfg, int mode, float temperature, uint64_t seed,
                                   uint64_t cycle, const void* target_logits, const int32_t* tokens,
                                   const int32_t* parent, const int32_t* n_tree, int32_t* accept_len,
                                   int32_t* accepted_slots, int32_t* out_tokens, void* stream) {
    struct Range {  // NVTX range over the call
        Range() { nvtxRangePushA("eagle_verify_static"); }
        ~Range() { nvtxRangePop(); }
    } range;
    if (cfg == nullptr) return EAGLE_ERR_INVALID_ARG;
    // Same checks as eagle_verify, through its public size query.
    if (eagle_workspace_bytes(cfg) == 0) return EAGLE_ERR_INVALID_ARG;
    if (mode != EAGLE_VERIFY_GREEDY && mode != EAGLE_VERIFY_LOSSLESS) return EAGLE_ERR_INVALID_ARG;
    const long rows = static_cast<long>(cfg->batch) * (cfg->node_budget + 1);
    if (cfg->batch > kMaxSeqs || rows > kMaxRows) return EAGLE_ERR_UNSUPPORTED;  // beyond the fixed scratch
    if (!target_logits || !tokens || !parent || !n_tree || !accept_len || !accepted_slots || !out_tokens)
        return EAGLE_ERR_INVALID_ARG;
    float inv_t = 1.0f;
    if (mode == EAGLE_VERIFY_LOSSLESS) {
        if (!(temperature > 0.0f) || !(temperature < INFINITY)) return EAGLE_ERR_INVALID_ARG;
        inv_t = static_cast<float>(1.0 / static_cast<double>(temperature));
    }
    if ((reinterpret_cast<uintptr_t>(target_logits) & 15u) != 0) return EAGLE_ERR_UNSUPPORTED;

    TreeDims d{};
    d.B = cfg->batch;
    d.V = cfg->vocab;
    d.k = cfg->top_k;
    d.D = cfg->depth;
    d.N = cfg->node_budget;
    d.T = cfg->node_budget + 1;
    d.W = (d.T + 31) / 32;
    d.C = cfg->top_k + (cfg->depth - 1) * cfg->top_k * cfg->top_k;
    d.log_thr = -INFINITY;  // not used by verification
    d.dtype = cfg->logit_dtype;
    d.policy = 0;  // not used by verification

    unsigned char* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return EAGLE_ERR_LAUNCH;
    TreeWs w{};
    w.status = reinterpret_cast<int*>(base + kOffStatus);
    w.verify_ticket = reinterpret_cast<int*>(base + kOffTicket);
    w.row_max = reinterpret_cast<float*>(base + kOffRowMax);
    w.row_arg = reinterpret_cast<int32_t*>(base + kOffRowArg);
    w.row_mass = reinterpret_cast<uint64_t*>(base + kOffRowMass);
    w.pmass = reinterpret_cast<uint64_t*>(base + kOffPMass);
    // The arrival counters and the status word must start at zero; the rest
    // is fully written by the kernels before it is read.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(base, 0, kOffTicket + d.B * sizeof(int), s) != cudaSuccess) return EAGLE_ERR_LAUNCH;
    const cudaError_t e = launch_verify(d, w, mode, inv_t, target_logits, tokens, parent, n_tree,
                                        verify_rng(seed, cycle), accept_len, accepted_slots, out_tokens, s);
    if (e != cudaSuccess) return EAGLE_ERR_LAUNCH;
#ifdef EAGLE_DEBUG
    // checked builds: wait (outside stream capture) and report the call's own device fault
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return EAGLE_ERR_LAUNCH;
        int v = 0;
        if (cudaMemcpy(&v, w.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return EAGLE_ERR_LAUNCH;
        if (v != 0) return v == 2 ? EAGLE_ERR_TIMEOUT : EAGLE_ERR_DEVICE;
    }
#endif
    return EAGLE_OK;
}
