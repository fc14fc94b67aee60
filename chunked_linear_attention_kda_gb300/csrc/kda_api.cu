// kda_api.cu -- the C ABI declared in include/kda.h: argument validation, kernel
// choice and launch, and the host-side schedule of the pipelined forward (its pieces, its
// streams and the one small kernel that writes the pieces' sequence offsets). Holds no
// arithmetic of the method.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstdio>
#include <string>
#include <vector>

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

// KDA_FWD_KERNEL=tc16 selects the 16-token-step mma.sync kernel instead of the 64-token-step
// tcgen05 kernel (same results within rounding; kept for side-by-side measurement)
bool use_tc16() {
    static const bool v = [] {
        const char *e = std::getenv("KDA_FWD_KERNEL");
        return e && std::string(e) == "tc16";
    }();
    return v;
}

kda_status run(const kda::FwdArgs &p, kda_dtype dtype, void *stream, Path path) {
    kda_status s = validate(p, dtype);
    if (s != KDA_OK) return s;
    if (p.n_seq == 0) return ok();
    cudaStream_t st = (cudaStream_t)stream;
    if (path == Path::kAuto && kda::fwd64_supported(p) && !use_tc16())
        return launched(kda::launch_fwd64(p, st), "tensor-core kernel launch");
    if (path == Path::kAuto && kda::tc_supported(p))
        return launched(kda::launch_tc(p, st), "tensor-core kernel launch");
    return launched(kda::launch_simt(p, st), "SIMT kernel launch");
}

// ---- pipelined forward from host memory -------------------------------------------------
//
// The token range is cut into segments; segment i's inputs are copied in on one stream
// while segment i-1 is computed on the caller's stream and segment i-2's outputs are copied
// out on a third. Each boundary is placed a multiple of 64 tokens after the start of the
// sequence that holds it, so every piece keeps its sequence's chunk grid, and the state of
// a sequence cut by a boundary is handed from one piece to the next in fp32 through the
// workspace: the result is the one the unsegmented call gives, bit for bit.

constexpr int kMaxSegments = 64;
// Cuts lie a multiple of this many tokens after their sequence's start: the serial step of
// the tensor-core kernel (64 tokens), itself a multiple of the SIMT kernel's 16-token chunk.
constexpr int64_t kStepGrid = 64;

// A piece: tokens [t0, t1) holding sequences [n0, n1) -- whole ones, or the part of one
// sequence that lies in a segment. Its start state is the caller's h0 rows n0.. (zeros
// without h0) or the carried state; its final state goes to the caller's h_final rows
// n0.. (nowhere without h_final) or to the carried state.
struct FwdPiece {
    int64_t t0, t1;
    int32_t n0, n1;
    int32_t h0_carried, hf_carried;
    int32_t segment;
};

// cu: host cu_seqlens, already checked (cu[0] = 0, non-decreasing, cu[n_seq] = n_tok).
void plan_pieces(const int32_t *cu, int32_t n_seq, int64_t n_tok, int32_t n_segments,
                 std::vector<FwdPiece> &out) {
    out.clear();
    std::vector<int64_t> bounds{0};
    for (int32_t i = 1; i < n_segments; ++i) {
        const int64_t b = n_tok * i / n_segments;
        if (b <= 0 || b >= n_tok) continue;
        // the sequence holding token b: the last n with cu[n] <= b (then cu[n + 1] > b)
        const int32_t n = (int32_t)(std::upper_bound(cu, cu + n_seq + 1, (int32_t)b) - cu) - 1;
        const int64_t at = cu[n] + (b - cu[n]) / kStepGrid * kStepGrid;
        if (at > bounds.back() && at < n_tok) bounds.push_back(at);
    }
    bounds.push_back(n_tok);
    int32_t n = 0;          // first sequence whose final state is not yet written
    bool carrying = false;  // sequence n started in an earlier segment
    for (size_t i = 0; i + 1 < bounds.size(); ++i) {
        const int64_t t0 = bounds[i], t1 = bounds[i + 1];
        const int32_t seg = (int32_t)i;
        if (carrying) {
            const bool beyond = cu[n + 1] > t1;
            out.push_back({t0, beyond ? t1 : (int64_t)cu[n + 1], n, n + 1, 1, beyond ? 1 : 0, seg});
            if (beyond) continue;
            ++n;
            carrying = false;
        }
        const int32_t c0 = n;
        while (n < n_seq && cu[n + 1] <= t1) ++n;
        if (n > c0) out.push_back({cu[c0], cu[n], c0, n, 0, 0, seg});
        if (n < n_seq && cu[n] < t1) {  // starts here, ends in a later segment
            out.push_back({cu[n], t1, n, n + 1, 0, 1, seg});
            carrying = true;
        }
    }
}

struct PieceTable {
    int32_t n0[3 * kMaxSegments], count[3 * kMaxSegments], off[3 * kMaxSegments];
    int32_t t0[3 * kMaxSegments], t1[3 * kMaxSegments];
    int32_t n_pieces;
};

// Piece j's cu_seqlens, relative to its first token: entry k = clamp(cu[n0 + k], t0, t1) - t0,
// k = 0 .. count (count = its number of sequences), written at table + off[j].
__global__ void piece_offsets_kernel(const int32_t *__restrict__ cu, int32_t *__restrict__ table,
                                     const PieceTable pt) {
    for (int j = 0; j < pt.n_pieces; ++j)
        for (int k = threadIdx.x; k <= pt.count[j]; k += blockDim.x)
            table[pt.off[j] + k] = min(max(cu[pt.n0[j] + k], pt.t0[j]), pt.t1[j]) - pt.t0[j];
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// The pipelined forward's two side streams and three events, made once per (host thread,
// device) and kept for the thread's lifetime (creating and destroying them on every call
// put driver work on the timed path); they are released with the CUDA context. Reusing
// them across calls is safe: each call starts both streams behind the caller's stream
// and ends by making the caller's stream wait for both.
struct SideStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
};

cudaError_t side_streams(SideStreams **out) {
    thread_local std::vector<std::pair<int, SideStreams>> per_device;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (auto &pd : per_device)
        if (pd.first == dev) {
            *out = &pd.second;
            return cudaSuccess;
        }
    SideStreams ss;
    e = cudaStreamCreateWithFlags(&ss.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ss.out, cudaStreamNonBlocking);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ss.ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        for (cudaEvent_t x : ss.ev) if (x) cudaEventDestroy(x);
        if (ss.in) cudaStreamDestroy(ss.in);
        if (ss.out) cudaStreamDestroy(ss.out);
        return e;
    }
    per_device.emplace_back(dev, ss);
    *out = &per_device.back().second;
    return cudaSuccess;
}

// gated forward: two carried states, the offset tables of up to kMaxSegments segments'
// pieces, and one slot of gate logits for a segment of up to seg_tokens + kStepGrid tokens
size_t gated_workspace(int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v, int32_t seg_tokens) {
    const size_t carry = align256((size_t)n_heads * d_k * d_v * 4);
    const size_t table = align256(((size_t)n_seq + 5 * (size_t)kMaxSegments + 1) * 4);
    const size_t slot = align256(((size_t)seg_tokens + kStepGrid) * n_heads * d_k * 4);
    return 2 * carry + table + slot;
}

size_t pipeline_workspace(int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v,
                          int32_t n_segments) {
    // two carried states, then the pieces' offset tables: at most 3 pieces per segment,
    // 2 entries for a piece of one cut sequence, count + 1 for a run of whole ones
    const size_t carry = align256((size_t)n_heads * d_k * d_v * 4);
    return 2 * carry + align256(((size_t)n_seq + 5 * (size_t)n_segments + 1) * 4);
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
        case KDA_ERR_NONFINITE: return "KDA_ERR_NONFINITE: non-finite values in the outputs";
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
    unsigned int f64 = 0;
    e = kda::read_fwd64_flags(&f64, reset != 0, (cudaStream_t)stream);
    if (e != cudaSuccess) return launched(e, "reading the device status word");
    *flags = v | g | bw | f64;
    return ok();
}

kda_status kda_validate_cu_seqlens(const int32_t *cu_seqlens, int32_t n_seq, int64_t n_tok,
                                   int32_t *d_status, void *stream) {
    if (!cu_seqlens || !d_status) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens and d_status are required");
    if (n_seq < 0 || n_tok < 0) return fail(KDA_ERR_INVALID_ARG, "n_seq and n_tok must be non-negative");
    if (((uintptr_t)cu_seqlens & 3u) || ((uintptr_t)d_status & 3u))
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens and d_status must be 4-byte aligned");
    return launched(kda::launch_validate_cu(cu_seqlens, n_seq, n_tok, d_status, (cudaStream_t)stream),
                    "validation kernel launch");
}

kda_status kda_count_nonfinite(const void *x, int64_t n, kda_dtype dtype, unsigned long long *d_count,
                               void *stream) {
    if ((!x && n > 0) || !d_count) return fail(KDA_ERR_INVALID_ARG, "x and d_count are required");
    if (n < 0) return fail(KDA_ERR_INVALID_ARG, "n must be non-negative");
    if (dtype != KDA_F32 && dtype != KDA_BF16)
        return fail(KDA_ERR_UNSUPPORTED, "dtype must be KDA_F32 or KDA_BF16");
    if (((uintptr_t)x & (dtype == KDA_BF16 ? 1u : 3u)) || ((uintptr_t)d_count & 7u))
        return fail(KDA_ERR_INVALID_ARG, "x or d_count misaligned");
    return launched(kda::launch_count_nonfinite(x, n, dtype == KDA_BF16, d_count, (cudaStream_t)stream),
                    "non-finite count launch");
}

kda_status kda_check_outputs(const void *out, int64_t n_out, kda_dtype dtype, const float *h_final,
                             int64_t n_h_final, unsigned long long *d_scratch, uint64_t *count,
                             void *stream) {
    if (!d_scratch || !count) return fail(KDA_ERR_INVALID_ARG, "d_scratch and count are required");
    if ((!out && n_out > 0) || (!h_final && n_h_final > 0) || n_out < 0 || n_h_final < 0)
        return fail(KDA_ERR_INVALID_ARG, "bad output pointer or size");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(d_scratch, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) return launched(e, "clearing the count");
    kda_status s = kda_count_nonfinite(out, n_out, dtype, d_scratch, stream);
    if (s != KDA_OK) return s;
    s = kda_count_nonfinite(h_final, n_h_final, KDA_F32, d_scratch, stream);
    if (s != KDA_OK) return s;
    unsigned long long host = 0;
    e = cudaMemcpyAsync(&host, d_scratch, sizeof(host), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return launched(e, "reading the count");
    *count = host;
    if (host > 0)
        return fail(KDA_ERR_NONFINITE, std::to_string(host) + " non-finite values in out / h_final");
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
    // the sizes are checked first, so the scratch comparison sees only valid ones
    kda_status s = validate(pack(q, k, v, gate_logits, beta, h0, cu_seqlens,
                                 const_cast<void *>(dout), nullptr, n_tok, n_seq, n_heads, d_k,
                                 d_v, dtype),
                            dtype);
    if (s != KDA_OK) return s;
    if (kda::bwd_workspace_bytes(n_tok, n_seq, n_heads, d_k, d_v) > kda::kStaticScratchBytes)
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

kda_status kda_gate_projection_out(const void *x, const void *weight, const float *bias, void *out,
                                   kda_dtype out_dtype, int64_t n_tok, int32_t d_model,
                                   int32_t n_out, void *stream) {
    if (out_dtype != KDA_F32 && out_dtype != KDA_BF16)
        return fail(KDA_ERR_UNSUPPORTED, "out_dtype must be KDA_F32 or KDA_BF16");
    if (!x || !weight || !out)
        return n_tok == 0 ? ok() : fail(KDA_ERR_INVALID_ARG, "x, weight and the output are required");
    if (n_tok < 0 || d_model <= 0 || n_out <= 0)
        return fail(KDA_ERR_INVALID_ARG, "n_tok must be >= 0, d_model and n_out positive");
    if (n_tok > 0x7fffffffLL) return fail(KDA_ERR_UNSUPPORTED, "n_tok above 2^31 - 1");
    if (d_model % 8 != 0)
        return fail(KDA_ERR_UNSUPPORTED, "d_model must be a multiple of 8 (16-byte rows for TMA)");
    const void *a16[] = {x, weight, out};
    for (const void *p : a16)
        if (!aligned16(p))
            return fail(KDA_ERR_INVALID_ARG, "x, weight and the output must be 16-byte aligned");
    if (((uintptr_t)bias & 3u) != 0) return fail(KDA_ERR_INVALID_ARG, "bias must be 4-byte aligned");
    const size_t es = out_dtype == KDA_BF16 ? 2 : 4;
    const uintptr_t o = (uintptr_t)out, ob = (uintptr_t)n_tok * n_out * es;
    struct Range { const void *p; size_t bytes; };
    const Range ins[] = {{x, (size_t)n_tok * d_model * 2}, {weight, (size_t)n_out * d_model * 2},
                         {bias, bias ? (size_t)n_out * 4 : 0}};
    for (const Range &r : ins)
        if (r.p && r.bytes && (uintptr_t)r.p < o + ob && o < (uintptr_t)r.p + r.bytes)
            return fail(KDA_ERR_INVALID_ARG, "the output may not overlap an input");
    if (n_tok == 0) return ok();
    const cudaError_t e =
        out_dtype == KDA_BF16
            ? kda::launch_gate_proj_bf16(x, weight, bias, out, (int)n_tok, n_out, d_model, (cudaStream_t)stream)
            : kda::launch_gate_proj(x, weight, bias, static_cast<float *>(out), (int)n_tok, n_out, d_model,
                                    (cudaStream_t)stream);
    return launched(e, "gate projection launch");
}

kda_status kda_gate_projection(const void *x, const void *weight, const float *bias,
                               float *gate_logits, int64_t n_tok, int32_t d_model,
                               int32_t n_out, void *stream) {
    return kda_gate_projection_out(x, weight, bias, gate_logits, KDA_F32, n_tok, d_model, n_out, stream);
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

size_t kda_chunk_fwd_pipelined_workspace_bytes(int32_t n_seq, int32_t n_heads, int32_t d_k,
                                               int32_t d_v, int32_t n_segments) {
    if (n_seq < 0 || n_heads <= 0 || d_k <= 0 || d_v <= 0 || n_segments < 1 ||
        n_segments > kMaxSegments)
        return 0;
    return pipeline_workspace(n_seq, n_heads, d_k, d_v, n_segments);
}

int32_t kda_chunk_fwd_pipeline_plan(const int32_t *host_cu_seqlens, int32_t n_seq,
                                    int64_t n_tok, int32_t n_segments, int64_t *pieces,
                                    int32_t capacity) {
    if (!host_cu_seqlens || n_seq < 0 || n_tok < 0 || n_segments < 1 ||
        n_segments > kMaxSegments || (n_tok > 0 && n_seq == 0) || n_tok > 0x7fffffffLL)
        return -1;
    if (n_seq > 0 && (host_cu_seqlens[0] != 0 || host_cu_seqlens[n_seq] != n_tok)) return -1;
    for (int32_t n = 0; n < n_seq; ++n)
        if (host_cu_seqlens[n + 1] < host_cu_seqlens[n]) return -1;
    std::vector<FwdPiece> plan;
    if (n_seq > 0) plan_pieces(host_cu_seqlens, n_seq, n_tok, n_segments, plan);
    if (pieces) {
        if ((int32_t)plan.size() > capacity) return -1;
        for (size_t j = 0; j < plan.size(); ++j) {
            int64_t *r = pieces + 7 * j;
            r[0] = plan[j].t0; r[1] = plan[j].t1; r[2] = plan[j].n0; r[3] = plan[j].n1;
            r[4] = plan[j].h0_carried; r[5] = plan[j].hf_carried; r[6] = plan[j].segment;
        }
    }
    return (int32_t)plan.size();
}

kda_status kda_chunk_fwd_from_host_pipelined(
    const void *host_q, const void *host_k, const void *host_v,
    const float *host_gate_logits, const float *host_beta, const float *host_h0,
    const int32_t *host_cu_seqlens, void *host_out, float *host_h_final, void *dev_q,
    void *dev_k, void *dev_v, float *dev_gate_logits, float *dev_beta, float *dev_h0,
    int32_t *dev_cu_seqlens, void *dev_out, float *dev_h_final, void *dev_workspace,
    size_t workspace_bytes, int64_t n_tok, int32_t n_seq, int32_t n_heads, int32_t d_k,
    int32_t d_v, int32_t n_segments, kda_dtype dtype, void *stream) {
    kda::FwdArgs whole = pack(dev_q, dev_k, dev_v, dev_gate_logits, dev_beta,
                              host_h0 ? dev_h0 : nullptr, dev_cu_seqlens, dev_out,
                              host_h_final ? dev_h_final : nullptr, n_tok, n_seq, n_heads, d_k,
                              d_v, dtype);
    kda_status s = validate(whole, dtype);
    if (s != KDA_OK) return s;
    if (n_segments < 1 || n_segments > kMaxSegments)
        return fail(KDA_ERR_INVALID_ARG, "n_segments must be in [1, 64]");
    if (n_seq > 0 && !host_cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "host_cu_seqlens is NULL");
    if (n_tok > 0 && (!host_q || !host_k || !host_v || !host_gate_logits || !host_beta ||
                      !host_out))
        return fail(KDA_ERR_INVALID_ARG, "host input/output pointers are required");
    if ((host_h0 && !dev_h0) || (host_h_final && !dev_h_final))
        return fail(KDA_ERR_INVALID_ARG, "a host state buffer needs its device buffer");
    if (n_seq > 0 && kda_chunk_fwd_pipeline_plan(host_cu_seqlens, n_seq, n_tok, 1, nullptr, 0) < 0)
        return fail(KDA_ERR_INVALID_ARG,
                    "host_cu_seqlens must start at 0, not decrease and end at n_tok (< 2^31)");
    const size_t need = pipeline_workspace(n_seq, n_heads, d_k, d_v, n_segments);
    if (!dev_workspace || workspace_bytes < need || ((uintptr_t)dev_workspace & 255u))
        return fail(KDA_ERR_INVALID_ARG, "dev_workspace must be 256-byte aligned and hold "
                                         "kda_chunk_fwd_pipelined_workspace_bytes bytes");
    if (n_seq == 0) return ok();
    const size_t es = dtype == KDA_BF16 ? 2 : 4;
    const size_t rk = (size_t)n_heads * d_k, rv = (size_t)n_heads * d_v;  // elements per token
    const size_t ns = (size_t)n_heads * d_k * d_v;                         // floats per sequence
    // a cut anywhere keeps every 16-byte-aligned tile of a piece aligned only if a token's
    // rows are whole multiples of 16 bytes; otherwise the call runs as one piece
    const bool cuttable = (rk * es) % 16 == 0 && (rv * es) % 16 == 0 && (rk * 4) % 16 == 0;
    std::vector<FwdPiece> plan;
    plan_pieces(host_cu_seqlens, n_seq, n_tok, cuttable ? n_segments : 1, plan);
    if (plan.empty() || plan.back().segment == 0)  // one segment: nothing to overlap
        return kda_chunk_fwd_from_host(host_q, host_k, host_v, host_gate_logits, host_beta,
                                       host_h0, host_cu_seqlens, host_out, host_h_final, dev_q,
                                       dev_k, dev_v, dev_gate_logits, dev_beta, dev_h0,
                                       dev_cu_seqlens, dev_out, dev_h_final, n_tok, n_seq,
                                       n_heads, d_k, d_v, dtype, stream);

    char *ws = static_cast<char *>(dev_workspace);
    const size_t carry_b = align256(ns * 4);
    float *carry[2] = {reinterpret_cast<float *>(ws), reinterpret_cast<float *>(ws + carry_b)};
    int32_t *table = reinterpret_cast<int32_t *>(ws + 2 * carry_b);
    PieceTable pt{};
    pt.n_pieces = (int32_t)plan.size();
    int32_t off = 0;
    for (size_t j = 0; j < plan.size(); ++j) {
        pt.n0[j] = plan[j].n0;
        pt.count[j] = plan[j].n1 - plan[j].n0;
        pt.t0[j] = (int32_t)plan[j].t0;
        pt.t1[j] = (int32_t)plan[j].t1;
        pt.off[j] = off;
        off += pt.count[j] + 1;
    }

    cudaStream_t st = (cudaStream_t)stream, s_in = nullptr, s_out = nullptr;
    cudaEvent_t *ev = nullptr;  // start, inputs landed, piece done
    {
        SideStreams *ss = nullptr;
        cudaError_t e = side_streams(&ss);
        if (e != cudaSuccess) return launched(e, "pipeline stream or event creation");
        s_in = ss->in;
        s_out = ss->out;
        ev = ss->ev;
    }
    cudaError_t e = cudaSuccess;
    // from here on, every return first makes the caller's stream wait for both side
    // streams, so nothing queued on them outlives the call's ordering
    auto finish = [&](kda_status r) {
        if (cudaEventRecord(ev[1], s_in) == cudaSuccess) cudaStreamWaitEvent(st, ev[1], 0);
        if (cudaEventRecord(ev[2], s_out) == cudaSuccess) cudaStreamWaitEvent(st, ev[2], 0);
        return r;
    };

    auto h2d = [&](void *dst, const void *src, size_t bytes) {
        return bytes ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s_in) : cudaSuccess;
    };
    auto d2h = [&](void *dst, const void *src, size_t bytes) {
        return bytes ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s_out) : cudaSuccess;
    };
    // both side streams start after the caller's earlier work (which may still read the
    // device buffers or the workspace)
    e = cudaEventRecord(ev[0], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev[0], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev[0], 0);
    if (e == cudaSuccess) e = h2d(dev_cu_seqlens, host_cu_seqlens, (size_t)(n_seq + 1) * 4);
    if (e == cudaSuccess) {
        piece_offsets_kernel<<<1, 256, 0, s_in>>>(dev_cu_seqlens, table, pt);
        e = cudaGetLastError();
        kda::count_launches(1);
    }
    if (e != cudaSuccess) return finish(launched(e, "pipeline set-up"));

    const char *hq = static_cast<const char *>(host_q), *hk = static_cast<const char *>(host_k);
    const char *hv = static_cast<const char *>(host_v);
    char *dq = static_cast<char *>(dev_q), *dk_ = static_cast<char *>(dev_k);
    char *dv_ = static_cast<char *>(dev_v), *dout = static_cast<char *>(dev_out);
    char *hout = static_cast<char *>(host_out);
    size_t j = 0;
    while (j < plan.size()) {
        const int32_t seg = plan[j].segment;
        size_t j1 = j;
        while (j1 < plan.size() && plan[j1].segment == seg) ++j1;
        const int64_t t0 = plan[j].t0, t1 = plan[j1 - 1].t1;
        // rows of h0 of the sequences that start in this segment; rows of h_final of the
        // sequences that end in it (both contiguous)
        int32_t r0 = n_seq, r1 = 0, f0 = n_seq, f1 = 0;
        for (size_t i = j; i < j1; ++i) {
            if (!plan[i].h0_carried) { r0 = std::min(r0, plan[i].n0); r1 = std::max(r1, plan[i].n1); }
            if (!plan[i].hf_carried) { f0 = std::min(f0, plan[i].n0); f1 = std::max(f1, plan[i].n1); }
        }
        const size_t nt = (size_t)(t1 - t0);
        if (host_h0 && r1 > r0)
            e = h2d(dev_h0 + (size_t)r0 * ns, host_h0 + (size_t)r0 * ns, (size_t)(r1 - r0) * ns * 4);
        if (e == cudaSuccess) e = h2d(dq + t0 * rk * es, hq + t0 * rk * es, nt * rk * es);
        if (e == cudaSuccess) e = h2d(dk_ + t0 * rk * es, hk + t0 * rk * es, nt * rk * es);
        if (e == cudaSuccess) e = h2d(dv_ + t0 * rv * es, hv + t0 * rv * es, nt * rv * es);
        if (e == cudaSuccess)
            e = h2d(dev_gate_logits + t0 * rk, host_gate_logits + t0 * rk, nt * rk * 4);
        if (e == cudaSuccess)
            e = h2d(dev_beta + t0 * n_heads, host_beta + t0 * n_heads, nt * n_heads * 4);
        if (e == cudaSuccess) e = cudaEventRecord(ev[1], s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[1], 0);
        if (e != cudaSuccess) return finish(launched(e, "pipeline host-to-device copy"));
        for (size_t i = j; i < j1; ++i) {
            const FwdPiece &pc = plan[i];
            const float *h0 = pc.h0_carried ? carry[seg & 1]
                              : host_h0     ? dev_h0 + (size_t)pc.n0 * ns : nullptr;
            float *hf = pc.hf_carried ? carry[(seg + 1) & 1]
                        : host_h_final ? dev_h_final + (size_t)pc.n0 * ns : nullptr;
            kda::FwdArgs p = pack(dq + pc.t0 * rk * es, dk_ + pc.t0 * rk * es,
                                  dv_ + pc.t0 * rv * es, dev_gate_logits + pc.t0 * rk,
                                  dev_beta + pc.t0 * n_heads, h0, table + pt.off[i],
                                  dout + pc.t0 * rv * es, hf, pc.t1 - pc.t0, pc.n1 - pc.n0,
                                  n_heads, d_k, d_v, dtype);
            s = run(p, dtype, stream, Path::kAuto);
            if (s != KDA_OK) return finish(s);
        }
        e = cudaEventRecord(ev[2], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev[2], 0);
        if (e == cudaSuccess) e = d2h(hout + t0 * rv * es, dout + t0 * rv * es, nt * rv * es);
        if (e == cudaSuccess && host_h_final && f1 > f0)
            e = d2h(host_h_final + (size_t)f0 * ns, dev_h_final + (size_t)f0 * ns,
                    (size_t)(f1 - f0) * ns * 4);
        if (e != cudaSuccess) return finish(launched(e, "pipeline device-to-host copy"));
        j = j1;
    }
    // the caller's stream continues after the last copy out
    e = cudaEventRecord(ev[0], s_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[0], 0);
    return finish(launched(e, "pipeline completion"));
}

size_t kda_chunk_fwd_gated_workspace_bytes(int32_t n_seq, int32_t n_heads, int32_t d_k,
                                           int32_t d_v, int32_t segment_tokens) {
    if (n_seq < 0 || n_heads <= 0 || d_k <= 0 || d_v <= 0 || segment_tokens < kStepGrid) return 0;
    return gated_workspace(n_seq, n_heads, d_k, d_v, segment_tokens);
}

kda_status kda_chunk_fwd_gated(const void *x, const void *w_gate, const float *b_gate,
                               int32_t d_model, const void *q, const void *k, const void *v,
                               const float *beta, const float *h0, const int32_t *cu_seqlens,
                               const int32_t *host_cu_seqlens, void *out, float *h_final,
                               void *workspace, size_t workspace_bytes, int64_t n_tok,
                               int32_t n_seq, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t segment_tokens, kda_dtype dtype, void *stream) {
    if (dtype != KDA_BF16)
        return fail(KDA_ERR_UNSUPPORTED, "the gated forward takes bf16 x, W and q, k, v");
    if (segment_tokens < kStepGrid)
        return fail(KDA_ERR_INVALID_ARG, "segment_tokens must be at least 64");
    // the forward's rules for the shared inputs (the workspace stands in for the gate logits)
    kda::FwdArgs whole = pack(q, k, v, static_cast<const float *>(workspace), beta, h0,
                              cu_seqlens, out, h_final, n_tok, n_seq, n_heads, d_k, d_v, dtype);
    kda_status s = validate(whole, dtype);
    if (s != KDA_OK) return s;
    if (d_model <= 0 || d_model % 8 != 0)
        return fail(KDA_ERR_UNSUPPORTED, "d_model must be a positive multiple of 8 (16-byte rows for TMA)");
    if (n_tok > 0 && (!x || !w_gate)) return fail(KDA_ERR_INVALID_ARG, "x and w_gate are required");
    if (!aligned16(x) || !aligned16(w_gate)) return fail(KDA_ERR_INVALID_ARG, "x and w_gate must be 16-byte aligned");
    if (((uintptr_t)b_gate & 3u) != 0) return fail(KDA_ERR_INVALID_ARG, "b_gate must be 4-byte aligned");
    if (n_seq > 0 && !host_cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "host_cu_seqlens is NULL");
    if (n_seq > 0 && kda_chunk_fwd_pipeline_plan(host_cu_seqlens, n_seq, n_tok, 1, nullptr, 0) < 0)
        return fail(KDA_ERR_INVALID_ARG,
                    "host_cu_seqlens must start at 0, not decrease and end at n_tok (< 2^31)");
    const size_t need = gated_workspace(n_seq, n_heads, d_k, d_v, segment_tokens);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
        return fail(KDA_ERR_INVALID_ARG, "workspace must be 256-byte aligned and hold "
                                         "kda_chunk_fwd_gated_workspace_bytes bytes");
    if (n_seq == 0 || n_tok == 0) {
        if (n_seq > 0 && h_final) {  // no token: every h_final row is its h0 row (or zero)
            const size_t bytes = (size_t)n_seq * n_heads * d_k * d_v * 4;
            const cudaError_t e = h0 ? cudaMemcpyAsync(h_final, h0, bytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream)
                                     : cudaMemsetAsync(h_final, 0, bytes, (cudaStream_t)stream);
            return launched(e, "empty gated forward");
        }
        return ok();
    }
    const size_t es = 2;
    const size_t rk = (size_t)n_heads * d_k, rv = (size_t)n_heads * d_v;  // elements per token
    const size_t ns = (size_t)n_heads * d_k * d_v;
    const bool cuttable = (rk * es) % 16 == 0 && (rv * es) % 16 == 0 && (rk * 4) % 16 == 0;
    const int64_t want = (n_tok + segment_tokens - 1) / segment_tokens;
    if (!cuttable && want > 1)
        return fail(KDA_ERR_UNSUPPORTED, "segments need token rows of whole 16-byte multiples");
    if (want > 0x7fffffffLL) return fail(KDA_ERR_INVALID_ARG, "too many segments");
    std::vector<FwdPiece> plan;
    plan_pieces(host_cu_seqlens, n_seq, n_tok, (int32_t)want, plan);
    const int64_t slot_tokens = (int64_t)segment_tokens + kStepGrid;

    char *ws = static_cast<char *>(workspace);
    const size_t carry_b = align256(ns * 4);
    float *carry[2] = {reinterpret_cast<float *>(ws), reinterpret_cast<float *>(ws + carry_b)};
    int32_t *table = reinterpret_cast<int32_t *>(ws + 2 * carry_b);
    float *slot = reinterpret_cast<float *>(ws + 2 * carry_b +
                                            align256(((size_t)n_seq + 5 * (size_t)kMaxSegments + 1) * 4));
    const cudaStream_t st = (cudaStream_t)stream;
    const char *xq = static_cast<const char *>(x);
    const char *cq = static_cast<const char *>(q), *ck = static_cast<const char *>(k);
    const char *cv = static_cast<const char *>(v);
    char *co = static_cast<char *>(out);
    size_t j = 0;
    while (j < plan.size()) {
        // a batch of up to kMaxSegments segments shares one offsets-kernel launch
        const int32_t seg0 = plan[j].segment;
        const size_t jbase = j;
        size_t jb = j;
        while (jb < plan.size() && plan[jb].segment < seg0 + kMaxSegments) ++jb;
        PieceTable pt{};
        pt.n_pieces = (int32_t)(jb - j);
        int32_t off = 0;
        for (size_t i = j; i < jb; ++i) {
            const size_t t = i - j;
            pt.n0[t] = plan[i].n0;
            pt.count[t] = plan[i].n1 - plan[i].n0;
            pt.t0[t] = (int32_t)plan[i].t0;
            pt.t1[t] = (int32_t)plan[i].t1;
            pt.off[t] = off;
            off += pt.count[t] + 1;
        }
        piece_offsets_kernel<<<1, 256, 0, st>>>(cu_seqlens, table, pt);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return launched(e, "gated forward set-up");
        kda::count_launches(1);
        while (j < jb) {
            const int32_t seg = plan[j].segment;
            size_t j1 = j;
            while (j1 < jb && plan[j1].segment == seg) ++j1;
            const int64_t t0 = plan[j].t0, t1 = plan[j1 - 1].t1;
            if (t1 - t0 > slot_tokens) return fail(KDA_ERR_INVALID_ARG, "a segment outgrew its slot");
            // this segment's gate logits, straight into the slot (kept small enough for L2)
            e = kda::launch_gate_proj(xq + (size_t)t0 * d_model * 2, w_gate, b_gate, slot,
                                      (int)(t1 - t0), (int)rk, d_model, st);
            if (e != cudaSuccess) return launched(e, "gate projection launch");
            for (size_t i = j; i < j1; ++i) {
                const FwdPiece &pc = plan[i];
                const float *ph0 = pc.h0_carried ? carry[seg & 1] : h0 ? h0 + (size_t)pc.n0 * ns : nullptr;
                float *phf = pc.hf_carried ? carry[(seg + 1) & 1] : h_final ? h_final + (size_t)pc.n0 * ns : nullptr;
                kda::FwdArgs p = pack(cq + pc.t0 * rk * es, ck + pc.t0 * rk * es, cv + pc.t0 * rv * es,
                                      slot + (size_t)(pc.t0 - t0) * rk, beta + pc.t0 * n_heads, ph0,
                                      table + pt.off[i - jbase], co + pc.t0 * rv * es, phf,
                                      pc.t1 - pc.t0, pc.n1 - pc.n0, n_heads, d_k, d_v, dtype);
                s = run(p, dtype, stream, Path::kAuto);
                if (s != KDA_OK) return s;
            }
            j = j1;
        }
    }
    return ok();
}

}  // extern "C"
