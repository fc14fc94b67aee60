// kda_api.cu -- the C ABI declared in include/kda.h: argument validation, kernel
// choice and launch. Holds no arithmetic of the method.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <string>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

kda_status fail(kda_status s, const std::string &why) {
    g_last_error = why;
    return s;
}

kda_status ok() {
    g_last_error.clear();
    return KDA_OK;
}

bool aligned16(const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

kda_status validate(const kda::FwdArgs &a, int dtype) {
    if (dtype != KDA_F32 && dtype != KDA_BF16)
        return fail(KDA_ERR_UNSUPPORTED, "dtype must be KDA_F32 or KDA_BF16");
    if (a.n_tok < 0 || a.n_seq < 0 || a.n_heads <= 0)
        return fail(KDA_ERR_INVALID_ARG, "n_tok and n_seq must be >= 0, n_heads > 0");
    if (a.d_k <= 0 || a.d_v <= 0)
        return fail(KDA_ERR_INVALID_ARG, "d_k and d_v must be positive");
    if (a.d_k > 128 || a.d_v > 128)
        return fail(KDA_ERR_UNSUPPORTED, "d_k and d_v above 128 are not built");
    if (a.n_tok > 0 && a.n_seq == 0)
        return fail(KDA_ERR_INVALID_ARG, "n_tok > 0 needs at least one sequence");
    if (a.n_seq > 0 && a.cu_seqlens == nullptr)
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (a.n_tok > 0 && (!a.q || !a.k || !a.v || !a.a || !a.beta || !a.out))
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, gate_logits, beta and out are required");
    if ((int64_t)a.n_seq * a.n_heads > 0x7fffffffLL)
        return fail(KDA_ERR_INVALID_ARG, "n_seq * n_heads exceeds 2^31 - 1");
    // tiles moved by TMA or 16-byte vector accesses need 16-byte alignment; the rest
    // are read and written as 4-byte scalars
    const void *tiles[] = {a.q, a.k, a.v, a.a, a.out};
    for (const void *p : tiles)
        if (!aligned16(p))
            return fail(KDA_ERR_INVALID_ARG, "q, k, v, gate_logits and out must be 16-byte aligned");
    const void *scalars[] = {a.beta, a.h0, a.cu_seqlens, a.h_final};
    for (const void *p : scalars)
        if (((uintptr_t)p & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "beta, h0, cu_seqlens and h_final must be 4-byte aligned");
    return KDA_OK;
}

kda::FwdArgs pack(const void *q, const void *k, const void *v, const float *a,
                  const float *beta, const float *h0, const int32_t *cu, void *out,
                  float *h_final, int64_t n_tok, int32_t n_seq, int32_t n_heads,
                  int32_t d_k, int32_t d_v, kda_dtype dtype) {
    kda::FwdArgs p;
    p.q = q; p.k = k; p.v = v; p.a = a; p.beta = beta; p.h0 = h0; p.cu_seqlens = cu;
    p.out = out; p.h_final = h_final;
    p.n_tok = n_tok; p.n_seq = n_seq; p.n_heads = n_heads; p.d_k = d_k; p.d_v = d_v;
    p.bf16 = dtype == KDA_BF16;
    return p;
}

kda_status launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess)
        return fail(KDA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    return ok();
}

enum class Path { kAuto, kSimt };

kda_status run(const kda::FwdArgs &p, kda_dtype dtype, void *stream, Path path) {
    kda_status s = validate(p, dtype);
    if (s != KDA_OK) return s;
    if (p.n_seq == 0) return ok();
    cudaStream_t st = (cudaStream_t)stream;
    if (path == Path::kAuto && kda::tc_supported(p))
        return launched(kda::launch_tc(p, st), "tensor-core kernel launch");
    return launched(kda::launch_simt(p, st), "SIMT kernel launch");
}

}  // namespace

namespace kda {
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace kda

extern "C" {

uint64_t kda_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int kda_version(void) { return 100; }

const char *kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: dtype or head dimension not built";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
    }
    return "unknown kda_status";
}

const char *kda_last_error(void) { return g_last_error.c_str(); }

kda_status kda_selftest_bounded_wait(int64_t limit_cycles, int32_t *d_returned, void *stream) {
    if (!d_returned || limit_cycles <= 0)
        return fail(KDA_ERR_INVALID_ARG, "d_returned must be non-NULL and the limit positive");
    return launched(kda::bounded_wait_selftest(limit_cycles, d_returned, (cudaStream_t)stream),
                    "self-test launch");
}

kda_status kda_read_device_flags(uint32_t *flags, int reset, void *stream) {
    if (!flags) return fail(KDA_ERR_INVALID_ARG, "flags is NULL");
    unsigned int v = 0, g = 0;
    cudaError_t e = kda::read_device_flags(&v, reset != 0, (cudaStream_t)stream);
    if (e != cudaSuccess) return launched(e, "reading the device status word");
    e = kda::read_gemm_flags(&g, reset != 0, (cudaStream_t)stream);
    if (e != cudaSuccess) return launched(e, "reading the device status word");
    unsigned int bw = 0;
    e = kda::read_bwd_flags(&bw, reset != 0, (cudaStream_t)stream);
    if (e != cudaSuccess) return launched(e, "reading the device status word");
    *flags = v | g | bw;
    return ok();
}

kda_status kda_affine_combine(const float *M, const float *S_in, const float *B, float *S_out,
                              int32_t n_heads, int32_t d_k, int32_t d_v, void *stream) {
    if (!M || !S_in || !B || !S_out)
        return fail(KDA_ERR_INVALID_ARG, "M, S_in, B and S_out are required");
    if (n_heads <= 0 || d_k <= 0 || d_v <= 0)
        return fail(KDA_ERR_INVALID_ARG, "n_heads, d_k and d_v must be positive");
    if (d_k > 128 || d_v > 128)
        return fail(KDA_ERR_UNSUPPORTED, "d_k and d_v above 128 are not built");
    const void *ptrs[] = {M, S_in, B, S_out};
    for (const void *p : ptrs)
        if (((uintptr_t)p & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "M, S_in, B and S_out must be 4-byte aligned");
    if (S_out == M || S_out == S_in || S_out == B)
        return fail(KDA_ERR_INVALID_ARG, "S_out may not alias an input");
    return launched(kda::launch_affine_combine(M, S_in, B, S_out, n_heads, d_k, d_v,
                                               (cudaStream_t)stream),
                    "affine combine launch");
}

kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *gate_logits, const float *beta, float *state, void *out,
                           int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v,
                           kda_dtype dtype, void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16)
        return fail(KDA_ERR_UNSUPPORTED, "dtype must be KDA_F32 or KDA_BF16");
    if (n_seq < 0 || n_heads <= 0)
        return fail(KDA_ERR_INVALID_ARG, "n_seq must be >= 0 and n_heads > 0");
    if (d_k <= 0 || d_v <= 0) return fail(KDA_ERR_INVALID_ARG, "d_k and d_v must be positive");
    if (d_k > 128 || d_v > 128)
        return fail(KDA_ERR_UNSUPPORTED, "d_k and d_v above 128 are not built");
    if ((int64_t)n_seq * n_heads > 0x7fffffffLL)
        return fail(KDA_ERR_INVALID_ARG, "n_seq * n_heads exceeds 2^31 - 1");
    if (n_seq == 0) return ok();
    if (!q || !k || !v || !gate_logits || !beta || !state || !out)
        return fail(KDA_ERR_INVALID_ARG, "every pointer is required");
    const size_t es = dtype == KDA_BF16 ? 2 : 4;
    const void *elems[] = {q, k, v, out};
    for (const void *p : elems)
        if (((uintptr_t)p % es) != 0)
            return fail(KDA_ERR_INVALID_ARG, "q, k, v and out must be aligned to their element size");
    const void *f32s[] = {gate_logits, beta, state};
    for (const void *p : f32s)
        if (((uintptr_t)p & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "gate_logits, beta and state must be 4-byte aligned");
    const size_t bh = (size_t)n_seq * n_heads;
    struct Range { const void *p; size_t bytes; };
    const Range ins[] = {{q, bh * d_k * es}, {k, bh * d_k * es}, {v, bh * d_v * es},
                         {gate_logits, bh * d_k * 4}, {beta, bh * 4}};
    const Range st_r = {state, bh * d_k * d_v * 4}, out_r = {out, bh * d_v * es};
    auto overlap = [](const Range &x, const Range &y) {
        const uintptr_t a = (uintptr_t)x.p, b = (uintptr_t)y.p;
        return a < b + y.bytes && b < a + x.bytes;
    };
    for (const Range &r : ins)
        if (overlap(r, st_r) || overlap(r, out_r))
            return fail(KDA_ERR_INVALID_ARG, "state and out may not overlap an input");
    if (overlap(st_r, out_r)) return fail(KDA_ERR_INVALID_ARG, "state and out may not overlap");
    kda::DecodeArgs p;
    p.q = q; p.k = k; p.v = v; p.a = gate_logits; p.beta = beta; p.state = state; p.out = out;
    p.n_seq = n_seq; p.n_heads = n_heads; p.d_k = d_k; p.d_v = d_v;
    p.bf16 = dtype == KDA_BF16;
    return launched(kda::launch_decode_step(p, (cudaStream_t)stream), "decode step launch");
}

size_t kda_chunk_bwd_workspace_bytes(int64_t n_tok, int32_t n_seq, int32_t n_heads,
                                     int32_t d_k, int32_t d_v) {
    if (n_tok < 0 || n_seq < 0 || n_heads <= 0 || d_k <= 0 || d_v <= 0) return 0;
    return kda::bwd_workspace_bytes(n_tok, n_seq, n_heads, d_k, d_v);
}

kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const float *gate_logits,
                         const float *beta, const float *h0, const int32_t *cu_seqlens,
                         const void *dout, const float *dh_final, void *dq, void *dk, void *dv,
                         float *dgate_logits, float *dbeta, float *dh0, void *workspace,
                         size_t workspace_bytes, int64_t n_tok, int32_t n_seq,
                         int32_t n_heads, int32_t d_k, int32_t d_v, kda_dtype dtype,
                         void *stream) {
    // the forward's argument rules for the shared inputs (out stands in for dout)
    kda_status s = validate(pack(q, k, v, gate_logits, beta, h0, cu_seqlens,
                                 const_cast<void *>(dout), nullptr, n_tok, n_seq, n_heads, d_k,
                                 d_v, dtype),
                            dtype);
    if (s != KDA_OK) return s;
    if (n_seq == 0) return ok();
    if (n_tok > 0 && (!dq || !dk || !dv || !dgate_logits || !dbeta))
        return fail(KDA_ERR_INVALID_ARG, "dq, dk, dv, dgate_logits and dbeta are required");
    const size_t need = kda::bwd_workspace_bytes(n_tok, n_seq, n_heads, d_k, d_v);
    if (!workspace || workspace_bytes < need)
        return fail(KDA_ERR_INVALID_ARG, "workspace is NULL or smaller than "
                                         "kda_chunk_bwd_workspace_bytes()");
    const size_t es = dtype == KDA_BF16 ? 2 : 4;
    const void *outs_io[] = {dq, dk, dv};
    for (const void *p : outs_io)
        if (((uintptr_t)p % es) != 0)
            return fail(KDA_ERR_INVALID_ARG, "dq, dk and dv must be aligned to their element size");
    const void *outs_f32[] = {dgate_logits, dbeta, dh0, dh_final, workspace};
    for (const void *p : outs_f32)
        if (((uintptr_t)p & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG,
                        "dgate_logits, dbeta, dh0, dh_final and workspace must be 4-byte aligned");
    struct Range { const void *p; size_t bytes; };
    const size_t nk = (size_t)n_tok * n_heads * d_k, nv = (size_t)n_tok * n_heads * d_v;
    const size_t ns = (size_t)n_seq * n_heads * d_k * d_v;
    const Range ins[] = {{q, nk * es}, {k, nk * es}, {v, nv * es}, {gate_logits, nk * 4},
                         {beta, (size_t)n_tok * n_heads * 4}, {h0, h0 ? ns * 4 : 0},
                         {dout, nv * es}, {dh_final, dh_final ? ns * 4 : 0},
                         {cu_seqlens, (size_t)(n_seq + 1) * 4}};
    const Range outs[] = {{dq, nk * es}, {dk, nk * es}, {dv, nv * es}, {dgate_logits, nk * 4},
                          {dbeta, (size_t)n_tok * n_heads * 4}, {dh0, dh0 ? ns * 4 : 0},
                          {workspace, need}};
    auto overlap = [](const Range &x, const Range &y) {
        if (!x.p || !y.p || !x.bytes || !y.bytes) return false;
        const uintptr_t a = (uintptr_t)x.p, b = (uintptr_t)y.p;
        return a < b + y.bytes && b < a + x.bytes;
    };
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        for (const Range &r : ins)
            if (overlap(outs[i], r))
                return fail(KDA_ERR_INVALID_ARG, "gradients and workspace may not overlap an input");
        for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
            if (overlap(outs[i], outs[j]))
                return fail(KDA_ERR_INVALID_ARG, "gradients and workspace may not overlap");
    }
    kda::BwdArgs p;
    p.q = q; p.k = k; p.v = v; p.dout = dout; p.a = gate_logits; p.beta = beta; p.h0 = h0;
    p.dh_final = dh_final; p.cu_seqlens = cu_seqlens; p.dq = dq; p.dk = dk; p.dv = dv;
    p.da = dgate_logits; p.dbeta = dbeta; p.dh0 = dh0; p.workspace = (float *)workspace;
    p.n_tok = n_tok; p.n_seq = n_seq; p.n_heads = n_heads; p.d_k = d_k; p.d_v = d_v;
    p.bf16 = dtype == KDA_BF16;
    return launched(kda::launch_bwd(p, (cudaStream_t)stream), "backward launch");
}

kda_status kda_bwd_timing_start(int capacity) {
    if (capacity < 1 || capacity > 1024)
        return fail(KDA_ERR_INVALID_ARG, "capacity must be in [1, 1024]");
    const cudaError_t e = kda::bwd_timing_start(capacity);
    if (e != cudaSuccess) return launched(e, "creating the timing events");
    return ok();
}

kda_status kda_bwd_timing_read(float *ms, int *calls) {
    if (!ms || !calls) return fail(KDA_ERR_INVALID_ARG, "ms and calls must not be NULL");
    const cudaError_t e = kda::bwd_timing_read(ms, calls);
    if (e != cudaSuccess) return launched(e, "reading the timing events");
    return ok();
}

kda_status kda_chunk_bwd_static_scratch(const void *q, const void *k, const void *v,
                                        const float *gate_logits, const float *beta,
                                        const float *h0, const int32_t *cu_seqlens,
                                        const void *dout, const float *dh_final, void *dq,
                                        void *dk, void *dv, float *dgate_logits, float *dbeta,
                                        float *dh0, int64_t n_tok, int32_t n_seq,
                                        int32_t n_heads, int32_t d_k, int32_t d_v,
                                        kda_dtype dtype, void *stream) {
    static_assert(KDA_STATIC_SCRATCH_BYTES == kda::kStaticScratchBytes, "one scratch size");
    if (n_tok >= 0 && n_seq >= 0 && n_heads > 0 && d_k > 0 && d_v > 0 &&
        kda::bwd_workspace_bytes(n_tok, n_seq, n_heads, d_k, d_v) > kda::kStaticScratchBytes)
        return fail(KDA_ERR_UNSUPPORTED, "the problem needs more checkpoint space than the "
                                         "static scratch holds (KDA_STATIC_SCRATCH_BYTES)");
    void *scratch = nullptr;
    if (n_seq > 0) {
        const cudaError_t e = kda::static_scratch(&scratch);
        if (e != cudaSuccess) return launched(e, "static scratch lookup");
    }
    return kda_chunk_bwd(q, k, v, gate_logits, beta, h0, cu_seqlens, dout, dh_final, dq, dk, dv,
                         dgate_logits, dbeta, dh0, scratch, kda::kStaticScratchBytes, n_tok,
                         n_seq, n_heads, d_k, d_v, dtype, stream);
}

kda_status kda_gate_projection(const void *x, const void *weight, const float *bias,
                               float *gate_logits, int64_t n_tok, int32_t d_model,
                               int32_t n_out, void *stream) {
    if (!x || !weight || !gate_logits)
        return n_tok == 0 ? ok() : fail(KDA_ERR_INVALID_ARG, "x, weight and gate_logits are required");
    if (n_tok < 0 || d_model <= 0 || n_out <= 0)
        return fail(KDA_ERR_INVALID_ARG, "n_tok must be >= 0, d_model and n_out positive");
    if (n_tok > 0x7fffffffLL) return fail(KDA_ERR_UNSUPPORTED, "n_tok above 2^31 - 1");
    if (d_model % 8 != 0)
        return fail(KDA_ERR_UNSUPPORTED, "d_model must be a multiple of 8 (16-byte rows for TMA)");
    const void *a16[] = {x, weight, gate_logits};
    for (const void *p : a16)
        if (!aligned16(p))
            return fail(KDA_ERR_INVALID_ARG, "x, weight and gate_logits must be 16-byte aligned");
    if (((uintptr_t)bias & 3u) != 0) return fail(KDA_ERR_INVALID_ARG, "bias must be 4-byte aligned");
    const uintptr_t o = (uintptr_t)gate_logits, ob = (uintptr_t)n_tok * n_out * 4;
    struct Range { const void *p; size_t bytes; };
    const Range ins[] = {{x, (size_t)n_tok * d_model * 2}, {weight, (size_t)n_out * d_model * 2},
                         {bias, bias ? (size_t)n_out * 4 : 0}};
    for (const Range &r : ins)
        if (r.p && r.bytes && (uintptr_t)r.p < o + ob && o < (uintptr_t)r.p + r.bytes)
            return fail(KDA_ERR_INVALID_ARG, "gate_logits may not overlap an input");
    if (n_tok == 0) return ok();
    return launched(kda::launch_gate_proj(x, weight, bias, gate_logits, (int)n_tok, n_out, d_model,
                                          (cudaStream_t)stream),
                    "gate projection launch");
}

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *gate_logits, const float *beta, const float *h0,
                         const int32_t *cu_seqlens, void *out, float *h_final,
                         int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
                         int32_t d_v, kda_dtype dtype, void *stream) {
    return run(pack(q, k, v, gate_logits, beta, h0, cu_seqlens, out, h_final, n_tok, n_seq,
                    n_heads, d_k, d_v, dtype),
               dtype, stream, Path::kAuto);
}

kda_status kda_chunk_fwd_variant(const void *q, const void *k, const void *v,
                                 const float *gate_logits, const float *beta, const float *h0,
                                 const int32_t *cu_seqlens, void *out, float *h_final,
                                 int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
                                 int32_t d_v, kda_dtype dtype, int32_t gate_kind,
                                 int32_t diag_path, void *stream) {
    if (gate_kind != KDA_GATE_BOUNDED && gate_kind != KDA_GATE_SOFTPLUS)
        return fail(KDA_ERR_INVALID_ARG, "gate_kind must be KDA_GATE_BOUNDED or KDA_GATE_SOFTPLUS");
    if (diag_path != KDA_DIAG_DENSE && diag_path != KDA_DIAG_PAIRS)
        return fail(KDA_ERR_INVALID_ARG, "diag_path must be KDA_DIAG_DENSE or KDA_DIAG_PAIRS");
    const kda::FwdArgs p = pack(q, k, v, gate_logits, beta, h0, cu_seqlens, out, h_final, n_tok,
                                n_seq, n_heads, d_k, d_v, dtype);
    kda_status s = validate(p, dtype);
    if (s != KDA_OK) return s;
    if (p.n_seq == 0) return ok();
    return launched(kda::launch_simt_variant(p, gate_kind, diag_path == KDA_DIAG_PAIRS,
                                             (cudaStream_t)stream),
                    "variant kernel launch");
}

kda_status kda_chunk_fwd_simt(const void *q, const void *k, const void *v,
                              const float *gate_logits, const float *beta,
                              const float *h0, const int32_t *cu_seqlens, void *out,
                              float *h_final, int64_t n_tok, int32_t n_seq,
                              int32_t n_heads, int32_t d_k, int32_t d_v, kda_dtype dtype,
                              void *stream) {
    return run(pack(q, k, v, gate_logits, beta, h0, cu_seqlens, out, h_final, n_tok, n_seq,
                    n_heads, d_k, d_v, dtype),
               dtype, stream, Path::kSimt);
}

kda_status kda_chunk_fwd_from_host(
    const void *host_q, const void *host_k, const void *host_v,
    const float *host_gate_logits, const float *host_beta, const float *host_h0,
    const int32_t *host_cu_seqlens, void *host_out, float *host_h_final, void *dev_q,
    void *dev_k, void *dev_v, float *dev_gate_logits, float *dev_beta, float *dev_h0,
    int32_t *dev_cu_seqlens, void *dev_out, float *dev_h_final, int64_t n_tok,
    int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v, kda_dtype dtype,
    void *stream) {
    kda::FwdArgs p = pack(dev_q, dev_k, dev_v, dev_gate_logits, dev_beta,
                          host_h0 ? dev_h0 : nullptr, dev_cu_seqlens, dev_out,
                          host_h_final ? dev_h_final : nullptr, n_tok, n_seq, n_heads, d_k,
                          d_v, dtype);
    kda_status s = validate(p, dtype);
    if (s != KDA_OK) return s;
    if (n_seq > 0 && !host_cu_seqlens)
        return fail(KDA_ERR_INVALID_ARG, "host_cu_seqlens is NULL");
    if (n_tok > 0 && (!host_q || !host_k || !host_v || !host_gate_logits || !host_beta ||
                      !host_out))
        return fail(KDA_ERR_INVALID_ARG, "host input/output pointers are required");
    if ((host_h0 && !dev_h0) || (host_h_final && !dev_h_final))
        return fail(KDA_ERR_INVALID_ARG, "a host state buffer needs its device buffer");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t es = dtype == KDA_BF16 ? 2 : 4;
    const size_t nk = (size_t)n_tok * n_heads * d_k, nv = (size_t)n_tok * n_heads * d_v;
    const size_t ns = (size_t)n_seq * n_heads * d_k * d_v;
    struct Copy { void *dst; const void *src; size_t bytes; };
    const Copy in[] = {{dev_q, host_q, nk * es},
                       {dev_k, host_k, nk * es},
                       {dev_v, host_v, nv * es},
                       {dev_gate_logits, host_gate_logits, nk * 4},
                       {dev_beta, host_beta, (size_t)n_tok * n_heads * 4},
                       {dev_h0, host_h0, host_h0 ? ns * 4 : 0},
                       {dev_cu_seqlens, host_cu_seqlens, n_seq > 0 ? (size_t)(n_seq + 1) * 4 : 0}};
    for (const Copy &c : in) {
        if (c.bytes == 0) continue;
        cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return launched(e, "host-to-device copy");
    }
    s = run(p, dtype, stream, Path::kAuto);
    if (s != KDA_OK) return s;
    if (nv > 0) {
        cudaError_t e = cudaMemcpyAsync(host_out, dev_out, nv * es, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return launched(e, "device-to-host copy");
    }
    if (host_h_final && ns > 0) {
        cudaError_t e = cudaMemcpyAsync(host_h_final, dev_h_final, ns * 4,
                                        cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return launched(e, "device-to-host copy");
    }
    return ok();
}

}  // extern "C"
