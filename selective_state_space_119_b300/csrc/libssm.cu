// libssm.cu -- the C ABI of libssm: argument validation, launch planning and
// dispatch. Declarations and the contract of every entry point are in
// include/ssm.h. No entry point allocates, frees, or synchronizes (except
// ssm_get_device_status, which is documented to synchronize).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "ssm.h"
#include "ssm_internal.h"
#include "ssm_tmap.h"

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int64_t kMaxDim = int64_t(1) << 31;     // per-axis limit
constexpr int64_t kMaxElems = int64_t(1) << 40;   // batch * seqlen * dim limit
// Planning. A CTA of the scan covers channels_per_cta channels of one batch
// row over one L-chunk, and an SM keeps several of them. Splitting the
// sequence into K chunks multiplies the CTAs by K, which fills more of the
// SMs, at the price of a chunk-state pass over every chunk but the last (about
// kStatePassCost of the output pass per token). The plan takes the K of least
// modelled time:
//   time ~ chunk_len * (wave_cost(output CTAs) + kStatePassCost * wave_cost(state CTAs))
// where wave_cost(n) sums, over the waves of n CTAs on the device's SMs, the
// cost of the busiest SM of the wave: 1 for one CTA, kTwoCtaCost for two. The
// constants are a fit to the measured chunk-count sweeps of the three bf16
// dstate-16 workloads on a B300 (the fastest measured counts: 37 chunks for b1
// L131072 d5120, 6 for b4 L2048 d1536, 8-16 for b8 L4096 d2048); the SM count
// is the current device's (148 when there is none, for host-side planning).
constexpr int64_t kResidentCtas = 2;
constexpr double kTwoCtaCost = 1.2;
constexpr double kStatePassCost = 0.4;
constexpr double kSplitCost = 0.0;
constexpr int64_t kMinChunk = 256;
constexpr int64_t kMaxChunks = 64;    // the range the sweeps measured

double wave_cost(int64_t ctas, int64_t sms) {
    const int64_t per_wave = sms * kResidentCtas;
    const int64_t full = ctas / per_wave, rem = ctas % per_wave;
    double c = double(full) * (kResidentCtas > 1 ? kTwoCtaCost : 1.0);
    if (rem > 0) c += rem > sms ? kTwoCtaCost : 1.0;
    return c;
}

int set_cuda(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t io_size(int32_t io) { return io == SSM_BF16 ? 2 : 4; }

bool valid_dstate(int64_t n) { return n == 1 || n == 2 || n == 4 || n == 8 || n == 16; }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int check_dims(const ssm_dims* d, bool scan) {
    if (!d) return SSM_ERR_NULL;
    if (d->io_dtype != SSM_F32 && d->io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (d->batch < 0 || d->dim < 0 || (scan && d->seqlen < 0)) return SSM_ERR_DIMS;
    if (!valid_dstate(d->dstate)) return SSM_ERR_DIMS;
    if (d->batch >= kMaxDim || d->dim >= kMaxDim || (scan && d->seqlen >= kMaxDim))
        return SSM_ERR_DIMS;
    if (scan && d->chunk_len_hint < 0) return SSM_ERR_DIMS;
    if (scan && (d->tile_config_hint < 0 || d->tile_config_hint > ssm::kScanTileConfigs))
        return SSM_ERR_DIMS;
    if (d->flags & ~(SSM_FLAG_ZOH | SSM_FLAG_BC_PER_CHANNEL)) return SSM_ERR_DIMS;
    const int64_t L = scan ? d->seqlen : 1;
    if (d->batch > 0 && d->dim > 0 && L > 0 &&
        (d->batch > kMaxElems / d->dim || d->batch * d->dim > kMaxElems / L))
        return SSM_ERR_DIMS;
    const int64_t vec = d->io_dtype == SSM_BF16 ? 8 : 4;
    if (d->dim % vec != 0) return SSM_ERR_ALIGN;
    return SSM_OK;
}

int choose_tile_cfg(int64_t N, int32_t hint) {
    if (N != 16) return 0;   // small dstate runs configuration 0 only
    if (hint > 0) return hint - 1;
    return 0;
}

// purpose: the forward (kPlanFwd) or the backward (kPlanBwd), whose chunk count
// follows its own rule (below).
constexpr int kPlanFwd = 0, kPlanBwd = 1;
// The backward's gradient pass holds three CTAs per SM, and a chunk more costs
// it little (its reverse-carry pass covers every chunk but the first whatever
// their number, and composing one more carry is 16 FMAs per channel), so its
// plan takes as many chunks as fill those slots in one wave (a chunk at least
// 64 tokens).
constexpr int64_t kBwdResidentCtas = 3;
constexpr int64_t kMinBwdChunk = 64;

int make_plan(const ssm_dims* d, ssm::ScanPlan* p, int purpose = kPlanFwd) {
    *p = ssm::ScanPlan{};
    const int64_t batch = d->batch, L = d->seqlen, dim = d->dim, N = d->dstate;
    const int64_t TS = ssm::kScanStageTokens;
    if (batch == 0 || L == 0 || dim == 0) return SSM_OK;
    p->tile_cfg = choose_tile_cfg(N, d->tile_config_hint);
    p->channels_per_cta = ssm::scan_tile_channels(p->tile_cfg);
    p->tiles = (dim + p->channels_per_cta - 1) / p->channels_per_cta;
    const int64_t per_chunk = p->tiles * batch;
    const int64_t sms = ssm::device_sms();
    int64_t chunk;
    if (d->chunk_len_hint > 0) {
        chunk = d->chunk_len_hint;
    } else if (purpose == kPlanBwd) {
        const int64_t k = std::max<int64_t>(
            1, std::min<int64_t>(kBwdResidentCtas * sms / per_chunk, L / kMinBwdChunk));
        chunk = (L + k - 1) / k;
    } else if (d->flags & SSM_FLAG_BC_PER_CHANNEL) {
        // per-channel B, C are bound by HBM: split the sequence until about 2.5
        // output CTAs per SM keep enough loads in flight (measured best for
        // b4 L2048 d1536: 8 chunks), chunks of at least 128 tokens
        const int64_t k = std::max<int64_t>(
            1, std::min<int64_t>((5 * sms / 2 + per_chunk - 1) / per_chunk, L / 128));
        chunk = ((L + k - 1) / k + TS - 1) / TS * TS;
    } else {
        // modelled time of every chunk count (see the planning note above)
        chunk = (L + TS - 1) / TS * TS;
        double best = double(chunk) * wave_cost(per_chunk, sms);
        const int64_t kmax = std::min<int64_t>(kMaxChunks, std::max<int64_t>(1, L / kMinChunk));
        for (int64_t k = 2; k <= kmax; ++k) {
            const int64_t c = ((L + k - 1) / k + TS - 1) / TS * TS;
            const int64_t nk = (L + c - 1) / c;
            const double t = double(c) * (wave_cost(per_chunk * nk, sms) +
                                          kStatePassCost * wave_cost(per_chunk * (nk - 1), sms)) +
                             kSplitCost;
            if (t < best) {
                best = t;
                chunk = c;
            }
        }
    }
    // whole pipeline stages per chunk, so that only the sequence end is ragged;
    // the backward's chunks need only start on a checkpoint (its blocks are
    // counted per chunk)
    const int64_t gran = purpose == kPlanBwd ? ssm::kCkptTokens : TS;
    chunk = std::max<int64_t>(gran, (chunk + gran - 1) / gran * gran);
    chunk = std::min(chunk, (L + gran - 1) / gran * gran);
    p->chunk_len = chunk;
    p->nchunks = (L + chunk - 1) / chunk;
    p->ctas = per_chunk * p->nchunks;
    if (p->ctas >= (int64_t(1) << 31)) return SSM_ERR_DIMS;
    p->kernels = p->nchunks > 1 ? 2 : 1;
    // header (status word) always; chunk carries when the sequence is split
    p->ws_bytes = ssm::kWsHeaderBytes;
    if (p->nchunks > 1) {
        const size_t carries = size_t(batch) * size_t(p->nchunks - 1) * size_t(dim);
        p->ws_off_H = ssm::kWsHeaderBytes;
        p->ws_off_S = p->ws_off_H + align256(carries * size_t(N) * sizeof(float));
        p->ws_bytes = p->ws_off_S + align256(carries * sizeof(float));
    }
    return SSM_OK;
}

struct Range {
    const void* p;
    size_t bytes;
};

bool overlap(const Range& a, const Range& b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

template <size_t NI, size_t NO>
int check_alias(const Range (&in)[NI], const Range (&out)[NO]) {
    for (size_t i = 0; i < NO; ++i) {
        for (size_t j = 0; j < NI; ++j)
            if (overlap(out[i], in[j])) return SSM_ERR_ALIAS;
        for (size_t j = i + 1; j < NO; ++j)
            if (overlap(out[i], out[j])) return SSM_ERR_ALIAS;
    }
    return SSM_OK;
}

template <size_t K>
int check_aligned(const void* const (&ptrs)[K]) {
    for (size_t i = 0; i < K; ++i)
        if (ptrs[i] && !aligned16(ptrs[i])) return SSM_ERR_ALIGN;
    return SSM_OK;
}

// Saved states of the checkpointing forward: the state before every
// kCkptTokens-th token, [batch][ceil(L / kCkptTokens)][dim][N] fp32.
size_t ckpt_bytes(const ssm_dims* d) {
    return size_t(d->batch) * size_t((d->seqlen + ssm::kCkptTokens - 1) / ssm::kCkptTokens) *
           size_t(d->dim) * size_t(d->dstate) * 4;
}

// Workspace of the backward: status header, the reverse chunk carries, and the
// per-CTA shares of the summed gradients (no dB | dC shares with per-channel
// rows: nothing sums over channels there).
struct BwdLayout {
    size_t off_Q = 0, off_S = 0, off_BC = 0, off_A = 0, off_D = 0, off_bias = 0, bytes = 0;
};

BwdLayout bwd_layout(const ssm_dims* d, const ssm::ScanPlan& p) {
    BwdLayout o;
    const size_t b = size_t(d->batch), L = size_t(d->seqlen), dim = size_t(d->dim);
    const size_t N = size_t(d->dstate), K = size_t(p.nchunks), tiles = size_t(p.tiles);
    size_t off = ssm::kWsHeaderBytes;
    if (K > 1) {
        o.off_Q = off;
        off += align256(b * (K - 1) * dim * N * 4);
        o.off_S = off;
        off += align256(b * (K - 1) * dim * 4);
    }
    o.off_BC = off;
    if (!(d->flags & SSM_FLAG_BC_PER_CHANNEL)) off += align256(b * tiles * L * 2 * N * 4);
    o.off_A = off;
    off += align256(b * K * dim * N * 4);
    o.off_D = off;
    off += align256(b * K * dim * 4);
    o.off_bias = off;
    off += align256(b * K * dim * 4);
    o.bytes = off;
    return o;
}

}  // namespace

extern "C" {

int ssm_version(void) { return (1 << 16) | 0; }

int ssm_last_cuda_error(void) { return g_last_cuda_error; }

const char* ssm_strerror(int code) {
    switch (code) {
        case SSM_OK: return "success";
        case SSM_ERR_NULL: return "a required pointer is NULL";
        case SSM_ERR_DIMS: return "invalid sizes (negative, too large, or unsupported dstate)";
        case SSM_ERR_DTYPE: return "io_dtype must be SSM_F32 or SSM_BF16";
        case SSM_ERR_ALIGN:
            return "pointer not 16-byte aligned, or dim not a multiple of 8 (bf16) / 4 (fp32)";
        case SSM_ERR_WORKSPACE: return "workspace missing or smaller than ssm_scan_workspace_bytes";
        case SSM_ERR_CUDA: return "a CUDA call failed (see ssm_last_cuda_error)";
        case SSM_ERR_TIMEOUT: return "device-side bounded wait gave up";
        case SSM_ERR_ALIAS: return "an output buffer overlaps an input";
        default: return "unknown libssm error code";
    }
}

int ssm_scan_plan(const ssm_dims* dims, ssm_plan* plan) {
    if (!plan) return SSM_ERR_NULL;
    int rc = check_dims(dims, true);
    if (rc != SSM_OK) return rc;
    ssm::ScanPlan p;
    rc = make_plan(dims, &p);
    if (rc != SSM_OK) return rc;
    plan->chunk_len = p.chunk_len;
    plan->nchunks = p.nchunks;
    plan->channels_per_cta = p.channels_per_cta;
    plan->ctas = p.ctas;
    plan->kernels = p.kernels;
    plan->tile_config = p.tile_cfg;
    return SSM_OK;
}

size_t ssm_scan_workspace_bytes(const ssm_dims* dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    ssm::ScanPlan p;
    if (make_plan(dims, &p) != SSM_OK) return 0;
    return p.ws_bytes;
}

}  // extern "C"

namespace {

// The conv taps of the fused input stage (NULL conv_w: no input stage).
struct ConvIn {
    const float* w = nullptr;
    const float* b = nullptr;
    int k = 0;
};

// The scan behind every scan entry point; h0 (state before the first token)
// may be NULL for h = 0; cv.w non-NULL puts the causal conv1d + SiLU in front.
int scan_impl(const void* x, const void* delta, const float* A, const void* B, const void* C,
              const float* D, const void* z, const float* delta_bias, int delta_softplus,
              const float* h0, void* out, float* final_state, const ssm_dims* dims,
              ssm_stream_t stream, const ConvIn& cv = ConvIn{}, float* ckpt = nullptr) {
    int rc = check_dims(dims, true);
    if (rc != SSM_OK) return rc;
    // the checkpointing forward feeds the backward, built for dstate 16 and
    // tile configuration 0
    if (ckpt && (dims->dstate != 16 || dims->tile_config_hint > 1)) return SSM_ERR_DIMS;
    // the fused input stage runs tile configuration 0 only
    if (cv.w && dims->dstate == 16 && dims->tile_config_hint > 1) return SSM_ERR_DIMS;
    // the exact zero-order hold is built for dstate 16, tile configuration 0,
    // without the fused input stage or checkpoints
    if ((dims->flags & SSM_FLAG_ZOH) && (dims->dstate != 16 || dims->tile_config_hint > 1 || cv.w))
        return SSM_ERR_DIMS;
    // so are per-channel B and C (and not with the exact zero-order hold)
    const bool bc_per_channel = (dims->flags & SSM_FLAG_BC_PER_CHANNEL) != 0;
    if (bc_per_channel && (dims->dstate != 16 || dims->tile_config_hint > 1 || cv.w ||
                           (dims->flags & SSM_FLAG_ZOH)))
        return SSM_ERR_DIMS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Empty problems: nothing to read (empty tensors may carry NULL pointers).
    if (dims->batch == 0 || dims->dim == 0) return SSM_OK;
    const size_t state_bytes = size_t(dims->batch) * dims->dim * dims->dstate * 4;
    if (dims->seqlen == 0) {
        // no token: the final state is the initial state
        if (!final_state) return SSM_OK;
        if (!aligned16(final_state) || (h0 && !aligned16(h0))) return SSM_ERR_ALIGN;
        if (h0 && overlap({h0, state_bytes}, {final_state, state_bytes})) return SSM_ERR_ALIAS;
        return set_cuda(h0 ? cudaMemcpyAsync(final_state, h0, state_bytes,
                                             cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(final_state, 0, state_bytes, s));
    }
    if (!x || !delta || !A || !B || !C || !out) return SSM_ERR_NULL;
    {
        const void* const ptrs[] = {x, delta, A, B, C, D, z, delta_bias, h0, out, final_state,
                                    dims->workspace, cv.w, cv.b, ckpt};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
    }
    ssm::ScanPlan p;
    rc = make_plan(dims, &p);
    if (rc != SSM_OK) return rc;
    if (p.ws_bytes > 0 && (!dims->workspace || dims->workspace_bytes < p.ws_bytes))
        return SSM_ERR_WORKSPACE;

    const int64_t batch = dims->batch, L = dims->seqlen, dim = dims->dim, N = dims->dstate;
    const size_t es = io_size(dims->io_dtype);
    const size_t elems = size_t(batch) * size_t(L) * size_t(dim);
    const size_t rows = size_t(batch) * size_t(L) * size_t(N) * (bc_per_channel ? size_t(dim) : 1);
    {
        const Range in[] = {{x, elems * es},      {delta, elems * es},
                            {z, elems * es},      {B, rows * es},
                            {C, rows * es},       {A, size_t(dim) * N * 4},
                            {D, size_t(dim) * 4}, {delta_bias, size_t(dim) * 4},
                            {h0, state_bytes},    {dims->workspace, p.ws_bytes},
                            {cv.w, size_t(dim) * size_t(cv.k) * 4},
                            {cv.b, size_t(dim) * 4}};
        const Range outs[] = {{out, elems * es},
                              {final_state, size_t(batch) * dim * N * 4},
                              {ckpt, size_t(batch) * size_t((L + ssm::kCkptTokens - 1) /
                                                            ssm::kCkptTokens) *
                                         size_t(dim) * size_t(N) * 4}};
        rc = check_alias(in, outs);
        if (rc != SSM_OK) return rc;
    }

    ssm::ScanArgs a{};
    a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.softplus = delta_softplus ? 1 : 0;
    a.h0 = h0;
    a.conv_w = cv.w; a.conv_b = cv.b; a.conv_k = cv.k;
    a.ckpt = ckpt; a.nckpt = (L + ssm::kCkptTokens - 1) / ssm::kCkptTokens;
    a.zoh = (dims->flags & SSM_FLAG_ZOH) ? 1 : 0;
    a.out = out; a.final_state = final_state;
    a.batch = batch; a.L = L; a.dim = dim;
    a.chunk_len = p.chunk_len; a.nchunks = p.nchunks; a.tiles = p.tiles;
    char* ws = static_cast<char*>(dims->workspace);
    a.status = reinterpret_cast<unsigned int*>(ws);
    if (p.nchunks > 1) {
        a.ws_H = reinterpret_cast<float*>(ws + p.ws_off_H);
        a.ws_S = reinterpret_cast<float*>(ws + p.ws_off_S);
    }
    if (bc_per_channel) return set_cuda(ssm::launch_scan_bcd(a, p, dims->io_dtype, s));
    // dstate 16 on the planner's own tile: the one-lane-per-channel kernel
    if (N == 16 && dims->tile_config_hint == 0 && !cv.w && !ckpt && !a.zoh)
        return set_cuda(ssm::launch_scan16(a, p, dims->io_dtype, s));
    return set_cuda(ssm::launch_scan(a, p, dims->io_dtype, static_cast<int>(N), s));
}

}  // namespace

namespace {

int check_ssd(const ssm_ssd_dims* d) {
    if (!d) return SSM_ERR_NULL;
    if (d->io_dtype != SSM_BF16) return d->io_dtype == SSM_F32 ? SSM_ERR_DIMS : SSM_ERR_DTYPE;
    if (d->batch < 0 || d->seqlen < 0 || d->nheads <= 0 || d->ngroups <= 0) return SSM_ERR_DIMS;
    if (d->headdim != 64 || d->dstate != 128 || d->nheads % d->ngroups != 0) return SSM_ERR_DIMS;
    if (d->flags != 0) return SSM_ERR_DIMS;
    if (d->batch >= kMaxDim || d->seqlen >= kMaxDim || d->nheads >= (int64_t(1) << 20))
        return SSM_ERR_DIMS;
    if (d->batch * d->nheads >= (int64_t(1) << 31)) return SSM_ERR_DIMS;
    if (d->batch > 0 && d->seqlen > 0 &&
        d->batch * d->seqlen > kMaxElems / (d->nheads * d->headdim))
        return SSM_ERR_DIMS;
    return SSM_OK;
}

}  // namespace

extern "C" {

int ssm_selective_scan_fwd(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* delta_bias, int delta_softplus, void* out,
                           float* final_state, const ssm_dims* dims, ssm_stream_t stream) {
    return scan_impl(x, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, out,
                     final_state, dims, stream);
}

int ssm_selective_scan_fwd_from_state(const void* x, const void* delta, const float* A,
                                      const void* B, const void* C, const float* D,
                                      const void* z, const float* delta_bias,
                                      int delta_softplus, const float* h0, void* out,
                                      float* final_state, const ssm_dims* dims,
                                      ssm_stream_t stream) {
    if (!h0 && dims && dims->batch > 0 && dims->dim > 0) return SSM_ERR_NULL;
    return scan_impl(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out,
                     final_state, dims, stream);
}

int ssm_selective_scan_fwd_conv(const void* x, const float* conv_w, const float* conv_b,
                                int conv_k, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z,
                                const float* delta_bias, int delta_softplus, void* out,
                                float* final_state, const ssm_dims* dims, ssm_stream_t stream) {
    if (conv_k < 1 || conv_k > ssm::kMaxConvK) return SSM_ERR_DIMS;
    if (!conv_w && dims && dims->batch > 0 && dims->dim > 0 && dims->seqlen > 0)
        return SSM_ERR_NULL;
    ConvIn cv;
    cv.w = conv_w; cv.b = conv_b; cv.k = conv_k;
    return scan_impl(x, delta, A, B, C, D, z, delta_bias, delta_softplus, nullptr, out,
                     final_state, dims, stream, cv);
}

size_t ssm_scan_checkpoint_bytes(const ssm_dims* dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->batch == 0 || dims->dim == 0 || dims->seqlen == 0) return 0;
    return ckpt_bytes(dims);
}

int ssm_selective_scan_fwd_ckpt(const void* x, const void* delta, const float* A, const void* B,
                                const void* C, const float* D, const void* z,
                                const float* delta_bias, int delta_softplus, const float* h0,
                                void* out, float* final_state, float* ckpt, const ssm_dims* dims,
                                ssm_stream_t stream) {
    if (!dims) return SSM_ERR_NULL;
    if (dims->dstate != 16 || dims->tile_config_hint > 1) return SSM_ERR_DIMS;
    if (!ckpt && dims->batch > 0 && dims->dim > 0 && dims->seqlen > 0) return SSM_ERR_NULL;
    return scan_impl(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, out, final_state,
                     dims, stream, ConvIn{}, ckpt);
}

size_t ssm_scan_bwd_workspace_bytes(const ssm_dims* dims) {
    if (check_dims(dims, true) != SSM_OK) return 0;
    if (dims->dstate != 16 || dims->tile_config_hint > 1) return 0;
    ssm::ScanPlan p;
    if (make_plan(dims, &p, kPlanBwd) != SSM_OK || p.nchunks == 0) return 0;
    return bwd_layout(dims, p).bytes;
}

int ssm_selective_scan_bwd(const void* x, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, const float* delta_bias,
                           int delta_softplus, const float* ckpt, const void* dout,
                           const float* dfinal_state, void* dx, void* ddelta, float* dA, void* dB,
                           void* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                           const ssm_dims* dims, ssm_stream_t stream) {
    int rc = check_dims(dims, true);
    if (rc != SSM_OK) return rc;
    // dstate 16, the planner's tile; either variant (the exact zero-order hold or
    // per-channel B and C), not both, as in the forward
    if (dims->dstate != 16 || dims->tile_config_hint > 1 ||
        ((dims->flags & SSM_FLAG_ZOH) && (dims->flags & SSM_FLAG_BC_PER_CHANNEL)))
        return SSM_ERR_DIMS;
    const bool bc_per_channel = (dims->flags & SSM_FLAG_BC_PER_CHANNEL) != 0;
    if (dims->batch == 0 || dims->dim == 0) return SSM_OK;
    if ((z == nullptr) != (dz == nullptr) && dims->seqlen > 0) return SSM_ERR_NULL;
    if (!dA) return SSM_ERR_NULL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t batch = dims->batch, L = dims->seqlen, dim = dims->dim, N = dims->dstate;
    const size_t state_bytes = size_t(batch) * size_t(dim) * size_t(N) * 4;
    if (L == 0) {
        // no token: the parameters get no gradient and dLoss/dh0 = dLoss/dfinal_state
        const void* const ptrs[] = {dA, dD, ddelta_bias, dh0, dfinal_state};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
        if (dh0 && dfinal_state && overlap({dh0, state_bytes}, {dfinal_state, state_bytes}))
            return SSM_ERR_ALIAS;
        rc = set_cuda(cudaMemsetAsync(dA, 0, size_t(dim) * size_t(N) * 4, s));
        if (rc == SSM_OK && dD) rc = set_cuda(cudaMemsetAsync(dD, 0, size_t(dim) * 4, s));
        if (rc == SSM_OK && ddelta_bias)
            rc = set_cuda(cudaMemsetAsync(ddelta_bias, 0, size_t(dim) * 4, s));
        if (rc == SSM_OK && dh0)
            rc = set_cuda(dfinal_state ? cudaMemcpyAsync(dh0, dfinal_state, state_bytes,
                                                         cudaMemcpyDeviceToDevice, s)
                                       : cudaMemsetAsync(dh0, 0, state_bytes, s));
        return rc;
    }
    if (!x || !delta || !A || !B || !C || !ckpt || !dout || !dx || !ddelta || !dB || !dC)
        return SSM_ERR_NULL;
    {
        const void* const ptrs[] = {x,  delta,  A,  B,  C,  D,  z,  delta_bias, ckpt, dout,
                                    dfinal_state, dx, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                                    dh0, dims->workspace};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
    }
    ssm::ScanPlan p;
    rc = make_plan(dims, &p, kPlanBwd);
    if (rc != SSM_OK) return rc;
    const BwdLayout lay = bwd_layout(dims, p);
    if (!dims->workspace || dims->workspace_bytes < lay.bytes) return SSM_ERR_WORKSPACE;
    {
        const size_t es = io_size(dims->io_dtype);
        const size_t elems = size_t(batch) * size_t(L) * size_t(dim);
        const size_t rows =
            size_t(batch) * size_t(L) * size_t(N) * (bc_per_channel ? size_t(dim) : 1);
        const Range in[] = {{x, elems * es},       {delta, elems * es},
                            {z, elems * es},       {dout, elems * es},
                            {B, rows * es},        {C, rows * es},
                            {A, size_t(dim) * N * 4}, {D, size_t(dim) * 4},
                            {delta_bias, size_t(dim) * 4}, {ckpt, ckpt_bytes(dims)},
                            {dfinal_state, state_bytes}};
        const Range outs[] = {{dx, elems * es},     {ddelta, elems * es},
                              {dz, elems * es},     {dB, rows * es},
                              {dC, rows * es},      {dA, size_t(dim) * N * 4},
                              {dD, size_t(dim) * 4}, {ddelta_bias, size_t(dim) * 4},
                              {dh0, state_bytes},   {dims->workspace, lay.bytes}};
        rc = check_alias(in, outs);
        if (rc != SSM_OK) return rc;
    }
    char* ws = static_cast<char*>(dims->workspace);
    ssm::BwdArgs a{};
    a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.softplus = delta_softplus ? 1 : 0;
    a.zoh = (dims->flags & SSM_FLAG_ZOH) ? 1 : 0;
    a.ckpt = ckpt; a.nckpt = (L + ssm::kCkptTokens - 1) / ssm::kCkptTokens;
    a.dout = dout; a.dfinal = dfinal_state;
    a.dx = dx; a.ddelta = ddelta; a.dz = dz; a.dh0 = dh0;
    a.dB = dB; a.dC = dC; a.dA = dA; a.dD = dD; a.dbias = ddelta_bias;
    a.batch = batch; a.L = L; a.dim = dim;
    a.chunk_len = p.chunk_len; a.nchunks = p.nchunks; a.tiles = p.tiles;
    if (p.nchunks > 1) {
        a.wsQ = reinterpret_cast<float*>(ws + lay.off_Q);
        a.wsS = reinterpret_cast<float*>(ws + lay.off_S);
    }
    a.pBC = bc_per_channel ? nullptr : reinterpret_cast<float*>(ws + lay.off_BC);
    a.pA = reinterpret_cast<float*>(ws + lay.off_A);
    a.pD = reinterpret_cast<float*>(ws + lay.off_D);
    a.pbias = reinterpret_cast<float*>(ws + lay.off_bias);
    if (bc_per_channel) return set_cuda(ssm::launch_scan_bcd_bwd(a, dims->io_dtype, s));
    return set_cuda(ssm::launch_scan_bwd(a, dims->io_dtype, s));
}

int ssm_causal_conv1d_silu(const void* x, const float* conv_w, const float* conv_b, int conv_k,
                           void* u, const ssm_dims* dims, ssm_stream_t stream) {
    if (!dims) return SSM_ERR_NULL;
    if (conv_k < 1 || conv_k > ssm::kMaxConvK) return SSM_ERR_DIMS;
    // only the [batch, seqlen, dim] sizes and io_dtype matter here
    ssm_dims d = *dims;
    d.dstate = 16; d.chunk_len_hint = 0; d.tile_config_hint = 0; d.flags = 0;
    int rc = check_dims(&d, true);
    if (rc != SSM_OK) return rc;
    if (d.batch == 0 || d.seqlen == 0 || d.dim == 0) return SSM_OK;
    if (!x || !conv_w || !u) return SSM_ERR_NULL;
    {
        const void* const ptrs[] = {x, conv_w, conv_b, u};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
    }
    const size_t elems = size_t(d.batch) * size_t(d.seqlen) * size_t(d.dim);
    {
        const Range in[] = {{x, elems * io_size(d.io_dtype)},
                            {conv_w, size_t(d.dim) * size_t(conv_k) * 4},
                            {conv_b, size_t(d.dim) * 4}};
        const Range outs[] = {{u, elems * io_size(d.io_dtype)}};
        rc = check_alias(in, outs);
        if (rc != SSM_OK) return rc;
    }
    ssm::ConvArgs a{};
    a.x = x; a.w = conv_w; a.b = conv_b; a.u = u;
    a.batch = d.batch; a.L = d.seqlen; a.dim = d.dim; a.k = conv_k;
    return set_cuda(ssm::launch_conv1d_silu(a, d.io_dtype,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

size_t ssm_causal_conv1d_silu_bwd_workspace_bytes(const ssm_dims* dims, int conv_k) {
    if (!dims || conv_k < 1 || conv_k > ssm::kMaxConvK) return 0;
    ssm_dims d = *dims;
    d.dstate = 16; d.chunk_len_hint = 0; d.tile_config_hint = 0; d.flags = 0;
    if (check_dims(&d, true) != SSM_OK) return 0;
    if (d.batch == 0 || d.seqlen == 0 || d.dim == 0) return 0;
    return ssm::kWsHeaderBytes +
           align256(ssm::conv1d_bwd_partial_floats(d.batch, d.seqlen, d.dim, conv_k) * 4);
}

int ssm_causal_conv1d_silu_bwd(const void* x, const float* conv_w, const float* conv_b,
                               int conv_k, const void* du, void* dx, float* dconv_w,
                               float* dconv_b, const ssm_dims* dims, ssm_stream_t stream) {
    if (!dims) return SSM_ERR_NULL;
    if (conv_k < 1 || conv_k > ssm::kMaxConvK) return SSM_ERR_DIMS;
    ssm_dims d = *dims;
    d.dstate = 16; d.chunk_len_hint = 0; d.tile_config_hint = 0; d.flags = 0;
    int rc = check_dims(&d, true);
    if (rc != SSM_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d.dim == 0) return SSM_OK;
    if (d.batch == 0 || d.seqlen == 0) {
        // no token: the weight and bias gradients are zero
        if (!dconv_w) return SSM_ERR_NULL;
        if (!aligned16(dconv_w) || (dconv_b && !aligned16(dconv_b))) return SSM_ERR_ALIGN;
        rc = set_cuda(cudaMemsetAsync(dconv_w, 0, size_t(d.dim) * conv_k * 4, s));
        if (rc == SSM_OK && dconv_b) rc = set_cuda(cudaMemsetAsync(dconv_b, 0, size_t(d.dim) * 4, s));
        return rc;
    }
    if (!x || !conv_w || !du || !dx || !dconv_w) return SSM_ERR_NULL;
    {
        const void* const ptrs[] = {x, conv_w, conv_b, du, dx, dconv_w, dconv_b, dims->workspace};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
    }
    const size_t need = ssm_causal_conv1d_silu_bwd_workspace_bytes(&d, conv_k);
    if (!dims->workspace || dims->workspace_bytes < need) return SSM_ERR_WORKSPACE;
    const size_t elems = size_t(d.batch) * size_t(d.seqlen) * size_t(d.dim);
    const size_t es = io_size(d.io_dtype);
    {
        const Range in[] = {{x, elems * es},
                            {conv_w, size_t(d.dim) * size_t(conv_k) * 4},
                            {conv_b, size_t(d.dim) * 4},
                            {du, elems * es},
                            {dims->workspace, need}};
        const Range outs[] = {{dx, elems * es},
                              {dconv_w, size_t(d.dim) * size_t(conv_k) * 4},
                              {dconv_b, size_t(d.dim) * 4}};
        rc = check_alias(in, outs);
        if (rc != SSM_OK) return rc;
    }
    ssm::ConvBwdArgs a{};
    a.x = x; a.w = conv_w; a.b = conv_b; a.du = du; a.dx = dx; a.dw = dconv_w; a.db = dconv_b;
    a.part = reinterpret_cast<float*>(static_cast<char*>(dims->workspace) + ssm::kWsHeaderBytes);
    a.batch = d.batch; a.L = d.seqlen; a.dim = d.dim; a.k = conv_k;
    return set_cuda(ssm::launch_conv1d_silu_bwd(a, d.io_dtype, s));
}

int ssm_state_update(float* state, const void* x, const void* delta, const float* A,
                     const void* B, const void* C, const float* D, const void* z,
                     const float* delta_bias, int delta_softplus, void* out,
                     const ssm_dims* dims, ssm_stream_t stream) {
    int rc = check_dims(dims, false);
    if (rc != SSM_OK) return rc;
    const bool bcd = (dims->flags & SSM_FLAG_BC_PER_CHANNEL) != 0;
    if (dims->batch == 0 || dims->dim == 0) return SSM_OK;   // nothing to update
    if (!state || !x || !delta || !A || !B || !C || !out) return SSM_ERR_NULL;
    {
        const void* const ptrs[] = {state, x, delta, A, B, C, D, z, delta_bias, out};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
    }
    const int64_t batch = dims->batch, dim = dims->dim, N = dims->dstate;
    const size_t es = io_size(dims->io_dtype);
    const size_t bd = size_t(batch) * size_t(dim);
    const size_t rows = (bcd ? bd : size_t(batch)) * size_t(N);   // B, C elements
    {
        const Range in[] = {{x, bd * es},          {delta, bd * es},
                            {z, bd * es},          {B, rows * es},
                            {C, rows * es},        {A, size_t(dim) * N * 4},
                            {D, size_t(dim) * 4},  {delta_bias, size_t(dim) * 4}};
        const Range outs[] = {{out, bd * es}, {state, bd * N * 4}};
        rc = check_alias(in, outs);
        if (rc != SSM_OK) return rc;
    }
    ssm::StepArgs a{};
    a.state = state; a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.softplus = delta_softplus ? 1 : 0; a.out = out;
    a.batch = batch; a.dim = dim;
    a.zoh = (dims->flags & SSM_FLAG_ZOH) ? 1 : 0;
    a.bc_per_channel = bcd ? 1 : 0;
    return set_cuda(ssm::launch_state_update(a, dims->io_dtype, static_cast<int>(N),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int ssm_debug_timeout_probe(void* workspace, size_t workspace_bytes, uint32_t max_polls,
                            ssm_stream_t stream) {
    if (!workspace) return SSM_ERR_NULL;
    if (workspace_bytes < ssm::kWsHeaderBytes) return SSM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SSM_ERR_ALIGN;
    if (max_polls < 1 || max_polls > (1u << 24)) return SSM_ERR_DIMS;
    return set_cuda(ssm::launch_timeout_probe(static_cast<unsigned int*>(workspace), max_polls,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

size_t ssm_ssd_workspace_bytes(const ssm_ssd_dims* dims) {
    return check_ssd(dims) == SSM_OK ? ssm::kWsHeaderBytes : 0;
}

int ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                const float* D, const float* dt_bias, int dt_softplus, const float* h0,
                void* y, float* final_state, const ssm_ssd_dims* dims, ssm_stream_t stream) {
    int rc = check_ssd(dims);
    if (rc != SSM_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t b = dims->batch, L = dims->seqlen, H = dims->nheads, G = dims->ngroups;
    const int64_t P = dims->headdim, N = dims->dstate;
    if (b == 0) return SSM_OK;
    const size_t state_bytes = size_t(b) * size_t(H) * size_t(P) * size_t(N) * 4;
    if (L == 0) {
        if (!final_state) return SSM_OK;
        if (!aligned16(final_state) || (h0 && !aligned16(h0))) return SSM_ERR_ALIGN;
        if (h0 && overlap({h0, state_bytes}, {final_state, state_bytes})) return SSM_ERR_ALIAS;
        return set_cuda(h0 ? cudaMemcpyAsync(final_state, h0, state_bytes,
                                             cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(final_state, 0, state_bytes, s));
    }
    if (!x || !dt || !A || !B || !C || !y) return SSM_ERR_NULL;
    {
        const void* const ptrs[] = {x, dt, A, B, C, D, dt_bias, h0, y, final_state,
                                    dims->workspace};
        rc = check_aligned(ptrs);
        if (rc != SSM_OK) return rc;
    }
    if (!dims->workspace || dims->workspace_bytes < ssm::kWsHeaderBytes) return SSM_ERR_WORKSPACE;
    const size_t xe = size_t(b) * size_t(L) * size_t(H) * size_t(P) * 2;
    const size_t re = size_t(b) * size_t(L) * size_t(G) * size_t(N) * 2;
    {
        const Range in[] = {{x, xe},
                            {dt, size_t(b) * size_t(L) * size_t(H) * 2},
                            {A, size_t(H) * 4},
                            {B, re},
                            {C, re},
                            {D, size_t(H) * 4},
                            {dt_bias, size_t(H) * 4},
                            {h0, state_bytes},
                            {dims->workspace, ssm::kWsHeaderBytes}};
        const Range outs[] = {{y, xe}, {final_state, state_bytes}};
        rc = check_alias(in, outs);
        if (rc != SSM_OK) return rc;
    }
    ssm::SsdLaunch l{};
    l.x = x; l.dt = dt; l.A = A; l.B = B; l.C = C; l.D = D; l.dt_bias = dt_bias;
    l.softplus = dt_softplus ? 1 : 0; l.h0 = h0; l.y = y; l.final_state = final_state;
    l.batch = b; l.L = L; l.H = H; l.G = G;
    l.status = static_cast<unsigned int*>(dims->workspace);
    return set_cuda(ssm::launch_ssd(l, s));
}

int ssm_ssd_get_device_status(const ssm_ssd_dims* dims, ssm_stream_t stream) {
    const int rc0 = check_ssd(dims);
    if (rc0 != SSM_OK) return rc0;
    int rc = set_cuda(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    if (rc != SSM_OK) return rc;
    if (!dims->workspace || dims->workspace_bytes < sizeof(uint32_t)) return SSM_ERR_WORKSPACE;
    uint32_t status = 0;
    rc = set_cuda(cudaMemcpy(&status, dims->workspace, sizeof(status), cudaMemcpyDeviceToHost));
    if (rc != SSM_OK) return rc;
    if (status != 0) {
        rc = set_cuda(cudaMemset(dims->workspace, 0, sizeof(status)));
        if (rc != SSM_OK) return rc;
    }
    return status == 0 ? SSM_OK : -static_cast<int>(status);
}

int ssm_get_device_status(const ssm_dims* dims, ssm_stream_t stream) {
    int rc = check_dims(dims, true);
    if (rc != SSM_OK) return rc;
    ssm::ScanPlan p;
    rc = make_plan(dims, &p);
    if (rc != SSM_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rc = set_cuda(cudaStreamSynchronize(s));
    if (rc != SSM_OK) return rc;
    if (p.ws_bytes == 0) return SSM_OK;
    if (!dims->workspace || dims->workspace_bytes < sizeof(uint32_t)) return SSM_ERR_WORKSPACE;
    uint32_t status = 0;
    rc = set_cuda(cudaMemcpy(&status, dims->workspace, sizeof(status), cudaMemcpyDeviceToHost));
    if (rc != SSM_OK) return rc;
    if (status != 0) {
        // the word is sticky: clear it now that it has been reported
        rc = set_cuda(cudaMemset(dims->workspace, 0, sizeof(status)));
        if (rc != SSM_OK) return rc;
    }
    return status == 0 ? SSM_OK : -static_cast<int>(status);
}

}  // extern "C"
