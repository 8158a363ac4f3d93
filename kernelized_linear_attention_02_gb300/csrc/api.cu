// api.cu -- the C ABI declared in include/linattn.h: argument checks,
// workspace sizing and kernel selection.  Every entry point validates all of
// its arguments before it enqueues anything.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "kernels.h"

namespace la {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace la

namespace {

thread_local std::string g_last_error;

la_status fail(la_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

la_status cuda_fail(cudaError_t e, const char* where) {
    return fail(LA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

enum class Call { kCausal, kNonCausal, kDecode, kState, kDelta };

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Checks every field of the parameter block and resolves it into a Problem.
la_status make_problem(const la_params* p, Call call, la::Problem* P) {
    if (!p) return fail(LA_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1) return fail(LA_ERR_INVALID_ARG, "batch must be >= 1 (got %lld)", (long long)p->batch);
    if (p->seq_len < 0) return fail(LA_ERR_INVALID_ARG, "seq_len must be >= 0");
    if (call == Call::kDecode && p->seq_len != 1)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step needs seq_len == 1 (got %lld)", (long long)p->seq_len);
    if (p->q_heads < 1 || p->kv_heads < 1) return fail(LA_ERR_INVALID_ARG, "head counts must be >= 1");
    if (p->q_heads % p->kv_heads != 0)
        return fail(LA_ERR_INVALID_ARG, "q_heads (%d) must be a multiple of kv_heads (%d)", p->q_heads,
                    p->kv_heads);
    if (p->key_dim < 1 || p->value_dim < 1) return fail(LA_ERR_INVALID_ARG, "key_dim and value_dim must be >= 1");
    if (p->key_dim > 128 || p->value_dim > 128)
        return fail(LA_ERR_UNSUPPORTED, "key_dim and value_dim above 128 are not implemented");
    if ((p->io_dtype != LA_F32 && p->io_dtype != LA_BF16) || (p->out_dtype != LA_F32 && p->out_dtype != LA_BF16))
        return fail(LA_ERR_INVALID_ARG, "io_dtype/out_dtype must be LA_F32 or LA_BF16 (floating point only)");
    if (p->feature_map < LA_FMAP_NONE || p->feature_map > LA_FMAP_RELU_EPS)
        return fail(LA_ERR_INVALID_ARG, "unknown feature_map %d", p->feature_map);
    if (p->use_normalizer != 0 && p->use_normalizer != 1)
        return fail(LA_ERR_INVALID_ARG, "use_normalizer must be 0 or 1");
    if (!std::isfinite(p->epsilon) || p->epsilon < 0.f) return fail(LA_ERR_INVALID_ARG, "epsilon must be finite and >= 0");
    if (!std::isfinite(p->scale)) return fail(LA_ERR_INVALID_ARG, "scale must be finite");
    if (p->update_rule < LA_RULE_LINEAR || p->update_rule > LA_RULE_GATED_DELTA)
        return fail(LA_ERR_INVALID_ARG, "unknown update_rule %d", p->update_rule);
    const bool delta = p->update_rule == LA_RULE_DELTA || p->update_rule == LA_RULE_GATED_DELTA;
    if (delta && call != Call::kDelta && call != Call::kState)
        return fail(LA_ERR_INVALID_ARG, "the delta rules take beta: call la_forward_causal_delta / la_decode_step_delta");
    if (!delta && call == Call::kDelta)
        return fail(LA_ERR_INVALID_ARG, "la_forward_causal_delta needs update_rule delta or gated_delta");
    if (delta && (p->feature_map != LA_FMAP_NONE || p->use_normalizer))
        return fail(LA_ERR_UNSUPPORTED, "the delta rules are defined without a feature map or normalizer");
    if (p->decay_per_key_dim != 0 && p->decay_per_key_dim != 1)
        return fail(LA_ERR_INVALID_ARG, "decay_per_key_dim must be 0 or 1");
    if (p->decay_per_key_dim && p->update_rule != LA_RULE_GATED && p->update_rule != LA_RULE_GATED_DELTA)
        return fail(LA_ERR_INVALID_ARG, "decay_per_key_dim needs a gated rule");
    if (p->update_rule == LA_RULE_GATED && (p->feature_map != LA_FMAP_NONE || p->use_normalizer))
        return fail(LA_ERR_UNSUPPORTED, "the gated rule is defined without a feature map or normalizer");
    if (call == Call::kNonCausal && p->update_rule != LA_RULE_LINEAR)
        return fail(LA_ERR_UNSUPPORTED, "non-causal attention has no decay (gated rule)");
    const int64_t grid = p->batch * (int64_t)p->kv_heads;
    if (grid > 0x7fffffff) return fail(LA_ERR_UNSUPPORTED, "batch * kv_heads too large");

    P->B = p->batch;
    P->T = p->seq_len;
    P->Hq = p->q_heads;
    P->Hkv = p->kv_heads;
    P->G = p->q_heads / p->kv_heads;
    P->Dk = p->key_dim;
    P->Dv = p->value_dim;
    P->io_bf16 = p->io_dtype == LA_BF16;
    P->out_bf16 = p->out_dtype == LA_BF16;
    P->fmap = p->feature_map;
    P->norm = p->use_normalizer;
    P->gated = p->update_rule == LA_RULE_GATED || p->update_rule == LA_RULE_GATED_DELTA;
    P->delta = delta;
    P->decay_dim = p->decay_per_key_dim;
    P->eps = p->epsilon;
    P->scale = p->scale == 0.f ? 1.f / std::sqrt((float)p->key_dim) : p->scale;
    return LA_OK;
}

size_t state_bytes(const la::Problem& P) { return sizeof(float) * (size_t)P.B * P.Hkv * P.Dk * P.Dv; }
size_t key_state_bytes(const la::Problem& P) { return sizeof(float) * (size_t)P.B * P.Hkv * P.Dk; }

size_t recurrent_need(const la::Problem& P, bool causal) {
    return causal ? la::recurrent_workspace_bytes(P) : round_up(state_bytes(P)) + round_up(key_state_bytes(P));
}

// Workspace that lets the call take its fastest path (la_workspace_bytes).
size_t workspace_bytes(const la::Problem& P, bool causal) {
    const size_t rec = recurrent_need(P, causal);
    if (causal && P.decay_dim) return std::max(rec, la::perdim_chunk_workspace_bytes(P));
    if (!la::chunk_supported(P)) return rec;
    return std::max(rec, la::chunk_workspace_bytes(P, causal));
}

// Smallest workspace the call accepts.  With one decay per key dimension
// that is the recurrence's: the tensor-core form runs when the workspace
// also holds its chunk tiles (workspace_bytes).
size_t required_workspace_bytes(const la::Problem& P, bool causal) {
    if (causal && P.decay_dim) return recurrent_need(P, causal);
    return workspace_bytes(P, causal);
}

la_status check_ws(const la::Problem& P, bool causal, void* ws, size_t ws_bytes) {
    const size_t need = required_workspace_bytes(P, causal);
    if (need == 0) return LA_OK;
    if (!ws || ws_bytes < need)
        return fail(LA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, ws ? ws_bytes : 0);
    if (reinterpret_cast<uintptr_t>(ws) % kAlign)
        return fail(LA_ERR_WORKSPACE, "workspace must be %zu-byte aligned", kAlign);
    return LA_OK;
}

// Scratch of la_forward_causal_noalloc: one buffer per device, part of the
// library's device image, so using it needs no allocation at call time.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// (cudaGetSymbolAddress, with the device current) on the first call per
// device and cached; a device reset gives the device a new context, and the
// first call in it looks the address up again.
cudaError_t noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[la::kMaxDevices] = {};
    static uint64_t ctx_of[la::kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= la::kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t ctx = la::current_context_id();
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev] || ctx == 0 || ctx_of[dev] != ctx) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = ptr;
        ctx_of[dev] = la::current_context_id();
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

int la_abi_version(void) { return LINATTN_ABI_VERSION; }

uint64_t la_launch_count(void) { return la::g_launches.load(std::memory_order_relaxed); }

unsigned la_device_error(int reset) { return la::chunk_device_error(reset != 0); }

la_status la_check_bounded_wait(uint32_t limit_us, la_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return fail(LA_ERR_INVALID_ARG, "limit_us must be in 1 .. 1000000");
    cudaError_t e = la::bounded_wait_selftest(limit_us, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "la_check_bounded_wait");
    g_last_error.clear();
    return LA_OK;
}

const char* la_last_error(void) { return g_last_error.c_str(); }

const char* la_status_string(la_status s) {
    switch (s) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARG: return "invalid argument";
    case LA_ERR_UNSUPPORTED: return "unsupported";
    case LA_ERR_WORKSPACE: return "workspace missing or too small";
    case LA_ERR_CUDA: return "CUDA error";
    case LA_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
    }
    return "unknown status";
}

const char* la_status_str(la_status s) { return la_status_string(s); }

la_status la_device_status(int reset) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "la_device_status");
    const unsigned w = la::chunk_device_error(reset != 0);
    if (w == ~0u) return fail(LA_ERR_CUDA, "la_device_status: the error word could not be read");
    if (w) return fail(LA_ERR_TIMEOUT, "bounded waits gave up: error word 0x%08x", w);
    g_last_error.clear();
    return LA_OK;
}

la_status la_get_initial_state(const la_params* p, float* S, float* Z, la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kState, &P);
    if (st != LA_OK) return st;
    if (!S) return fail(LA_ERR_INVALID_ARG, "S is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(S, 0, state_bytes(P), s);
    if (e == cudaSuccess && Z) e = cudaMemsetAsync(Z, 0, key_state_bytes(P), s);
    if (e != cudaSuccess) return cuda_fail(e, "la_get_initial_state");
    g_last_error.clear();
    return LA_OK;
}

size_t la_workspace_bytes(const la_params* p, int causal) {
    la::Problem P;
    if (make_problem(p, causal ? Call::kCausal : Call::kNonCausal, &P) != LA_OK) return 0;
    return workspace_bytes(P, causal != 0);
}

la_status la_forward_causal_masked(const la_params* p, const void* q, const void* k, const void* v,
                                   const void* decay, const uint8_t* mask, const float* S0, const float* Z0,
                                   void* y, float* S_out, float* Z_out, void* ws, size_t ws_bytes,
                                   la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kCausal, &P);
    if (st != LA_OK) return st;
    P.mask = mask;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!P.norm) Z0 = nullptr, Z_out = nullptr;  // no key_state without the normalizer
    if (P.T == 0) {  // nothing to attend: the state passes through
        cudaError_t e = cudaSuccess;
        if (S_out && S_out != S0)
            e = S0 ? cudaMemcpyAsync(S_out, S0, state_bytes(P), cudaMemcpyDeviceToDevice, s)
                   : cudaMemsetAsync(S_out, 0, state_bytes(P), s);
        if (e == cudaSuccess && Z_out && Z_out != Z0)
            e = Z0 ? cudaMemcpyAsync(Z_out, Z0, key_state_bytes(P), cudaMemcpyDeviceToDevice, s)
                   : cudaMemsetAsync(Z_out, 0, key_state_bytes(P), s);
        if (e != cudaSuccess) return cuda_fail(e, "la_forward_causal");
        g_last_error.clear();
        return LA_OK;
    }
    if (!q || !k || !v || !y) return fail(LA_ERR_INVALID_ARG, "q, k, v and y are required when seq_len > 0");
    if (P.gated && !decay) return fail(LA_ERR_INVALID_ARG, "the gated rule needs decay");
    if ((st = check_ws(P, true, ws, ws_bytes)) != LA_OK) return st;
    cudaError_t e;
    // per-key-dimension decay: its own tensor-core form when the workspace
    // holds its chunk tiles, else the CUDA-core recurrence
    const size_t pd_need = P.decay_dim ? la::perdim_chunk_workspace_bytes(P) : 0;
    if (!P.decay_dim && la::chunk_supported(P) && la::chunk_pointers_ok(q, k, v, y))
        e = la::chunk_causal(P, q, k, v, P.gated ? decay : nullptr, S0, Z0, y, S_out, Z_out, ws, s);
    else if (pd_need > 0 && ws && ws_bytes >= pd_need && la::chunk_pointers_ok(q, k, v, y) &&
             reinterpret_cast<uintptr_t>(decay) % 16 == 0)
        e = la::perdim_chunk_causal(P, q, k, v, decay, S0, y, S_out, ws, s);
    else
        e = la::recurrent_causal(P, q, k, v, P.gated ? decay : nullptr, S0, Z0, y, S_out, Z_out, s, ws, ws_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "la_forward_causal");
    g_last_error.clear();
    return LA_OK;
}

la_status la_forward_causal(const la_params* p, const void* q, const void* k, const void* v,
                            const void* decay, const float* S0, const float* Z0, void* y,
                            float* S_out, float* Z_out, void* ws, size_t ws_bytes, la_stream_t stream) {
    return la_forward_causal_masked(p, q, k, v, decay, nullptr, S0, Z0, y, S_out, Z_out, ws, ws_bytes, stream);
}

la_status la_forward_causal_noalloc(const la_params* p, const void* q, const void* k, const void* v,
                                    const void* decay, const float* S0, const float* Z0, void* y,
                                    float* S_out, float* Z_out, la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kCausal, &P);
    if (st != LA_OK) return st;
    if (P.T == 0) return la_forward_causal(p, q, k, v, decay, S0, Z0, y, S_out, Z_out, nullptr, 0, stream);
    // the fastest path that fits the scratch (with one decay per key
    // dimension the recurrence when the tensor-core tiles do not fit)
    const size_t full = workspace_bytes(P, true);
    const size_t need = full <= LA_NOALLOC_SCRATCH_BYTES ? full : required_workspace_bytes(P, true);
    if (need > LA_NOALLOC_SCRATCH_BYTES)
        return fail(LA_ERR_WORKSPACE,
                    "la_forward_causal_noalloc: this problem needs %zu bytes of scratch, more than the %zu "
                    "built in; call la_forward_causal with a workspace instead",
                    need, (size_t)LA_NOALLOC_SCRATCH_BYTES);
    void* ws = nullptr;
    if (need > 0) {
        cudaError_t e = noalloc_scratch(&ws);
        if (e != cudaSuccess) return cuda_fail(e, "la_forward_causal_noalloc: scratch address");
    }
    return la_forward_causal(p, q, k, v, decay, S0, Z0, y, S_out, Z_out, ws, need > 0 ? LA_NOALLOC_SCRATCH_BYTES : 0,
                             stream);
}

la_status la_forward_noncausal_masked(const la_params* p, const void* q, const void* k, const void* v,
                                      const uint8_t* mask, void* y, void* ws, size_t ws_bytes,
                                      la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kNonCausal, &P);
    if (st != LA_OK) return st;
    P.mask = mask;
    if (P.T == 0) {
        g_last_error.clear();
        return LA_OK;
    }
    if (!q || !k || !v || !y) return fail(LA_ERR_INVALID_ARG, "q, k, v and y are required when seq_len > 0");
    if ((st = check_ws(P, false, ws, ws_bytes)) != LA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (la::chunk_supported(P) && la::chunk_pointers_ok(q, k, v, y)) {
        e = la::chunk_noncausal(P, q, k, v, y, ws, s);
    } else {
        float* S_ws = static_cast<float*>(ws);
        float* Z_ws = reinterpret_cast<float*>(static_cast<char*>(ws) + round_up(state_bytes(P)));
        e = la::recurrent_noncausal(P, q, k, v, y, S_ws, Z_ws, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "la_forward_noncausal");
    g_last_error.clear();
    return LA_OK;
}

la_status la_forward_noncausal(const la_params* p, const void* q, const void* k, const void* v, void* y,
                               void* ws, size_t ws_bytes, la_stream_t stream) {
    return la_forward_noncausal_masked(p, q, k, v, nullptr, y, ws, ws_bytes, stream);
}

la_status la_decode_step_masked(const la_params* p, const void* q, const void* k, const void* v,
                                const void* decay, const uint8_t* mask, float* S, float* Z, void* y,
                                la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kDecode, &P);
    if (st != LA_OK) return st;
    P.mask = mask;
    if (!q || !k || !v || !y || !S) return fail(LA_ERR_INVALID_ARG, "q, k, v, y and S are required");
    if (P.norm && !Z) return fail(LA_ERR_INVALID_ARG, "Z is required when use_normalizer = 1");
    if (P.gated && !decay) return fail(LA_ERR_INVALID_ARG, "the gated rule needs decay");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (la::decode_supported(P) && reinterpret_cast<uintptr_t>(S) % 16 == 0)
        e = la::decode_step(P, q, k, v, P.gated ? decay : nullptr, S, P.norm ? Z : nullptr, y, s);
    else
        e = la::recurrent_causal(P, q, k, v, P.gated ? decay : nullptr, S, P.norm ? Z : nullptr, y, S,
                                 P.norm ? Z : nullptr, s);
    if (e != cudaSuccess) return cuda_fail(e, "la_decode_step");
    g_last_error.clear();
    return LA_OK;
}

la_status la_decode_step(const la_params* p, const void* q, const void* k, const void* v, const void* decay,
                         float* S, float* Z, void* y, la_stream_t stream) {
    return la_decode_step_masked(p, q, k, v, decay, nullptr, S, Z, y, stream);
}

size_t la_backward_workspace_bytes(const la_params* p) {
    la::Problem P;
    if (make_problem(p, Call::kCausal, &P) != LA_OK) return 0;
    return la::backward_workspace_bytes(P);
}

la_status la_backward_causal(const la_params* p, const void* q, const void* k, const void* v, const float* S0,
                             const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0, float* dZ0,
                             void* ws, size_t ws_bytes, la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kCausal, &P);
    if (st != LA_OK) return st;
    if (P.gated) return fail(LA_ERR_UNSUPPORTED, "la_backward_causal covers the linear rule only");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!P.norm) Z0 = nullptr, dZ0 = nullptr;
    if (P.T == 0) {  // no tokens: the initial state's gradient is zero
        cudaError_t e = cudaSuccess;
        if (dS0) e = cudaMemsetAsync(dS0, 0, state_bytes(P), s);
        if (e == cudaSuccess && dZ0) e = cudaMemsetAsync(dZ0, 0, key_state_bytes(P), s);
        if (e != cudaSuccess) return cuda_fail(e, "la_backward_causal");
        g_last_error.clear();
        return LA_OK;
    }
    if (!q || !k || !v || !dy || !dq || !dk || !dv)
        return fail(LA_ERR_INVALID_ARG, "q, k, v, dy, dq, dk and dv are required when seq_len > 0");
    const size_t need = la::backward_workspace_bytes(P);
    if (!ws || ws_bytes < need)
        return fail(LA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, ws ? ws_bytes : 0);
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(LA_ERR_WORKSPACE, "workspace must be %zu-byte aligned", kAlign);
    cudaError_t e = la::backward_causal(P, q, k, v, S0, Z0, dy, dq, dk, dv, dS0, dZ0, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "la_backward_causal");
    g_last_error.clear();
    return LA_OK;
}

la_status la_forward_causal_delta(const la_params* p, const void* q, const void* k, const void* v,
                                  const void* decay, const void* beta, int beta_per_head, const uint8_t* mask,
                                  const float* S0, void* y, float* S_out, la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kDelta, &P);
    if (st != LA_OK) return st;
    if (beta_per_head != 0 && beta_per_head != 1) return fail(LA_ERR_INVALID_ARG, "beta_per_head must be 0 or 1");
    P.mask = mask;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (P.T == 0) {  // the state passes through
        cudaError_t e = cudaSuccess;
        if (S_out && S_out != S0)
            e = S0 ? cudaMemcpyAsync(S_out, S0, state_bytes(P), cudaMemcpyDeviceToDevice, s)
                   : cudaMemsetAsync(S_out, 0, state_bytes(P), s);
        if (e != cudaSuccess) return cuda_fail(e, "la_forward_causal_delta");
        g_last_error.clear();
        return LA_OK;
    }
    if (!q || !k || !v || !y || !beta) return fail(LA_ERR_INVALID_ARG, "q, k, v, beta and y are required");
    if (P.gated && !decay) return fail(LA_ERR_INVALID_ARG, "gated_delta needs decay");
    cudaError_t e = la::recurrent_delta(P, q, k, v, P.gated ? decay : nullptr, beta, beta_per_head, S0, y, S_out, s);
    if (e != cudaSuccess) return cuda_fail(e, "la_forward_causal_delta");
    g_last_error.clear();
    return LA_OK;
}

size_t la_delta_workspace_bytes(const la_params* p) {
    la::Problem P;
    if (make_problem(p, Call::kDelta, &P) != LA_OK) return 0;
    return la::delta_chunk_workspace_bytes(P);
}

la_status la_forward_causal_delta_ws(const la_params* p, const void* q, const void* k, const void* v,
                                     const void* decay, const void* beta, int beta_per_head, const uint8_t* mask,
                                     const float* S0, void* y, float* S_out, void* ws, size_t ws_bytes,
                                     la_stream_t stream) {
    la::Problem P;
    la_status st = make_problem(p, Call::kDelta, &P);
    if (st != LA_OK) return st;
    if (beta_per_head != 0 && beta_per_head != 1) return fail(LA_ERR_INVALID_ARG, "beta_per_head must be 0 or 1");
    P.mask = mask;
    const size_t need = la::delta_chunk_workspace_bytes(P);
    if (P.T == 0 || need == 0)  // no chunk form for this shape: the recurrence, which needs no workspace
        return la_forward_causal_delta(p, q, k, v, decay, beta, beta_per_head, mask, S0, y, S_out, stream);
    if (!q || !k || !v || !y || !beta) return fail(LA_ERR_INVALID_ARG, "q, k, v, beta and y are required");
    if (P.gated && !decay) return fail(LA_ERR_INVALID_ARG, "gated_delta needs decay");
    if (!ws || ws_bytes < need)
        return fail(LA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, ws ? ws_bytes : 0);
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(LA_ERR_WORKSPACE, "workspace must be %zu-byte aligned", kAlign);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (la::chunk_pointers_ok(q, k, v, y))
        e = la::delta_chunk_causal(P, q, k, v, P.gated ? decay : nullptr, beta, beta_per_head, S0, y, S_out, ws, s);
    else
        e = la::recurrent_delta(P, q, k, v, P.gated ? decay : nullptr, beta, beta_per_head, S0, y, S_out, s);
    if (e != cudaSuccess) return cuda_fail(e, "la_forward_causal_delta_ws");
    g_last_error.clear();
    return LA_OK;
}

la_status la_decode_step_delta(const la_params* p, const void* q, const void* k, const void* v,
                               const void* decay, const void* beta, int beta_per_head, const uint8_t* mask,
                               float* S, void* y, la_stream_t stream) {
    if (p && p->seq_len != 1)
        return fail(LA_ERR_INVALID_ARG, "la_decode_step_delta needs seq_len == 1 (got %lld)", (long long)p->seq_len);
    if (!S) return fail(LA_ERR_INVALID_ARG, "S is required");
    return la_forward_causal_delta(p, q, k, v, decay, beta, beta_per_head, mask, S, y, S, stream);
}

}  // extern "C"
