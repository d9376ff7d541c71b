// abi.cu -- the C ABI of libgdn.so (declared in include/gdn.h): argument
// validation, launch geometry and dispatch.  Validation happens entirely on
// the host, before any CUDA call, and follows the error rules of
// dispatch_repeat_tiled_f32 ("mlx-native repeat_tiled.rs"): zero dimensions,
// a head count that does not divide, size products that overflow and buffers
// that are too small are invalid arguments.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "gdn.h"
#include "launch.h"
#include "record.cuh"
#include "record_mma.cuh"
#include "replay.cuh"
#include "chunk.cuh"

namespace {

thread_local std::string g_last_error;

gdn_status fail(gdn_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

gdn_status ok() {
    g_last_error.clear();
    return GDN_OK;
}

bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }

// Product of dims (all > 0) times elem_bytes, or -1 on overflow.
int64_t nbytes(std::initializer_list<int64_t> dims, int64_t elem_bytes) {
    int64_t acc = elem_bytes;
    for (int64_t d : dims)
        if (!mul_ok(acc, d, &acc)) return -1;
    return acc;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

int elem_bytes(gdn_dtype dt) {
    switch (dt) {
    case GDN_DTYPE_F32: return 4;
    case GDN_DTYPE_BF16: return 2;
    case GDN_DTYPE_F16: return 2;
    }
    return 0;
}

gdn_status cuda_fail(const char *fn, const char *what, cudaError_t e) {
    return fail(GDN_ERR_CUDA, "%s: %s: %s (%s)", fn, what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// SM count of the current device (0 if it cannot be read).
int current_sm_count(cudaError_t *err) {
    int dev = 0, sms = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Testing hooks (gdn_force_launch_failures, gdn_set_wait_bound).
constexpr long long kDefaultWaitBound = 2000000000ll;  // clock cycles, about a second
std::atomic<int> g_forced_failures{0};
std::atomic<long long> g_wait_bound{kDefaultWaitBound};
std::atomic<int> g_inject_expiry{0};

// Consume one forced failure, if any is pending.
bool take_forced_failure() {
    int n = g_forced_failures.load();
    while (n > 0)
        if (g_forced_failures.compare_exchange_weak(n, n - 1)) return true;
    return false;
}

gdn_status forced_failure(const char *fn) {
    return cuda_fail(fn, "launch (forced by gdn_force_launch_failures)", cudaErrorLaunchFailure);
}

}  // namespace

namespace gdn {

long long wait_bound_cycles() { return g_wait_bound.load(); }
int inject_wait_expiry() { return g_inject_expiry.load(); }

bool supported_dk(int64_t dk) {
    return dk == 32 || dk == 64 || dk == 128 || dk == 192 || dk == 256;
}

int rows_per_warp(int dk) {
    switch (dk) {
    case 32: return DefaultLayout<32>::type::RW;
    case 64: return DefaultLayout<64>::type::RW;
    case 128: return DefaultLayout<128>::type::RW;
    case 192: return DefaultLayout<192>::type::RW;
    case 256: return DefaultLayout<256>::type::RW;
    }
    return 0;
}

static int max_warps(int dk) {
    switch (dk) {
    case 32: return DefaultLayout<32>::type::MAX_WARPS;
    case 64: return DefaultLayout<64>::type::MAX_WARPS;
    case 128: return DefaultLayout<128>::type::MAX_WARPS;
    case 192: return DefaultLayout<192>::type::MAX_WARPS;
    case 256: return DefaultLayout<256>::type::MAX_WARPS;
    }
    return 1;
}

// Warps per CTA: at most max_w (kMaxWarpsPerCta, launch.h, by default),
// fewer (rows of a tile split over more CTAs) when the tiles are few.
static int pick_warps(int dk, int rw, int64_t tiles, int64_t Dv, int sm_count,
                      int max_w = kMaxWarpsPerCta) {
    int nw = (int)std::min<int64_t>(std::min(max_warps(dk), max_w), ceil_div(Dv, rw));
    const int64_t want = 2 * (int64_t)(sm_count > 0 ? sm_count : 1);
    while (nw > 1 && tiles * ceil_div(Dv, (int64_t)nw * rw) < want) nw = (nw + 1) / 2;
    return nw;
}

static constexpr int kChunk = 16;        // timesteps staged in shared memory at a time
static constexpr int kMmaMinSteps = 12;  // shortest call routed to the mma.sync chunk kernel
// Shortest call routed to the tcgen05 record kernel (where it is eligible).
// Its time hardly depends on the call's length (22.6-23.6 us at B = 16,
// 58.6-59.5 us at B = 64 for 2 to 11 steps, Hv = 32, Dk = Dv = 128), while
// the FP32 kernel's grows with every step: 22.3 against 22.7 us at 6 steps,
// 24.5 against 22.7 at 8, 26.7 against 23.6 at 11.
static constexpr int kTcMinSteps = 7;

Geometry record_geometry(int dk, int64_t tiles, int64_t Dv, int64_t T, int esize, bool bf16,
                         int sm_count) {
    // the tensor-core chunk kernel pays for its 16-step chunk machinery only
    // when calls carry enough steps; short calls take the FP32 kernel
    if (bf16 && record_mma_supported(dk) && T >= kMmaMinSteps) {
        Geometry g;
        g.threads = 32 * kMmaWarps;
        g.rows_cta = kMmaRows;
        g.row_blocks = ceil_div(Dv, g.rows_cta);
        g.tc = kMmaChunk;
        g.smem = record_mma_smem_bytes(dk);
        g.mma = true;
        return g;
    }
    // a single step (decode) is all load and store: two-warp CTAs, twice as
    // many of them, schedule finer (measured 8 % faster at B = 32, Dk = 128;
    // eight steps and more are faster with four)
    const int rw = rows_per_warp(dk);
    const int nw = pick_warps(dk, rw, tiles, Dv, sm_count, T == 1 ? 2 : kMaxWarpsPerCta);
    Geometry g;
    g.threads = 32 * nw;
    g.rows_cta = nw * rw;
    g.row_blocks = ceil_div(Dv, g.rows_cta);
    g.tc = (int)std::min<int64_t>(T, kChunk);
    g.smem = record_smem_bytes(dk, g.tc, g.rows_cta, esize);
    g.mma = false;
    return g;
}

Geometry replay_geometry(int dk, int64_t tiles, int64_t Dv, int64_t steps, int esize, int sm_count) {
    const int rw = rows_per_warp(dk);
    const int nw = pick_warps(dk, rw, tiles, Dv, sm_count);
    Geometry g;
    g.threads = 32 * nw;
    g.rows_cta = nw * rw;
    g.row_blocks = ceil_div(Dv, g.rows_cta);
    g.tc = (int)std::max<int64_t>(1, std::min<int64_t>(steps, kChunk));
    g.smem = replay_smem_bytes(dk, g.tc, g.rows_cta, esize);
    g.mma = false;
    return g;
}

}  // namespace gdn

extern "C" {

const char *gdn_status_string(gdn_status status) {
    switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARGUMENT: return "GDN_ERR_INVALID_ARGUMENT";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    }
    return "GDN_ERR_UNKNOWN";
}

const char *gdn_last_error(void) { return g_last_error.c_str(); }

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

gdn_status gdn_wait_status(int *expired) {
    if (!expired) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_wait_status: expired must be non-NULL");
    unsigned rec = 0, rep = 0, str = 0;
    cudaError_t e = gdn::record_tc_take_wait_flag(&rec);
    if (e != cudaSuccess) return cuda_fail("gdn_wait_status", "record flag", e);
    e = gdn::replay_tc_take_wait_flag(&rep);
    if (e != cudaSuccess) return cuda_fail("gdn_wait_status", "replay flag", e);
    e = gdn::replay_stream_take_wait_flag(&str);
    if (e != cudaSuccess) return cuda_fail("gdn_wait_status", "stream replay flag", e);
    *expired = (rec | rep | str) != 0u ? 1 : 0;
    return ok();
}

gdn_status gdn_set_wait_bound(int64_t cycles) {
    if (cycles < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_set_wait_bound: cycles (%lld) must be >= 0",
                    (long long)cycles);
    g_wait_bound.store(cycles == 0 ? kDefaultWaitBound : (long long)cycles);
    return ok();
}

gdn_status gdn_inject_wait_expiry(int on) {
    g_inject_expiry.store(on != 0 ? 1 : 0);
    return ok();
}

gdn_status gdn_force_launch_failures(int n) {
    if (n < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_force_launch_failures: n (%d) must be >= 0", n);
    g_forced_failures.store(n);
    return ok();
}

}  // extern "C"

namespace {

gdn_status record_impl(const char *fn, const void *q, const void *k, const void *v, const void *g,
                       const void *beta, const void *state_in, const uint32_t *mask, void *y,
                       void *state_out, void *delta_log, void *k_log, void *g_log, int64_t B,
                       int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                       gdn_gqa_mapping mapping, gdn_dtype dtype, bool tstate, gdn_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(GDN_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dtype);
    if (mapping != GDN_GQA_BLOCK && mapping != GDN_GQA_TILED)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: unknown GQA mapping %d", fn, (int)mapping);
    if (B <= 0 || T <= 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: B, T, Hk, Hv, Dk, Dv must all be > 0 (got %lld %lld %lld %lld %lld %lld)", fn,
                    (long long)B, (long long)T, (long long)Hk, (long long)Hv, (long long)Dk, (long long)Dv);
    if (Hv % Hk != 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: Hv (%lld) must be a multiple of Hk (%lld)", fn,
                    (long long)Hv, (long long)Hk);
    if (!q || !k || !v || !g || !beta || !state_in || !y || !state_out || !delta_log)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: q, k, v, g, beta, state_in, y, state_out, delta_log must be non-NULL", fn);
    if (Dk % 32 != 0 || !gdn::supported_dk(Dk))
        return fail(GDN_ERR_UNSUPPORTED, "%s: Dk = %lld not supported (32, 64, 128, 192, 256)", fn,
                    (long long)Dk);
    const int64_t qk_b = nbytes({B, T, Hk, Dk}, eb), v_b = nbytes({B, T, Hv, Dv}, eb);
    const int64_t s_b = nbytes({B, Hv, Dv, Dk}, tstate ? eb : 4), kl_b = nbytes({B, T, Hv, Dk}, eb);
    const int64_t gb_b = nbytes({B, T, Hv}, eb), m_b = nbytes({B, T}, 4);
    if (qk_b < 0 || v_b < 0 || s_b < 0 || kl_b < 0 || gb_b < 0 || m_b < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: tensor sizes overflow int64", fn);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(state_in, 16) || !aligned(state_out, 16) ||
        !aligned(k_log, 16))
        return fail(GDN_ERR_MISALIGNED, "%s: q, k, state_in, state_out, k_log must be 16-byte aligned",
                    fn);
    if (!aligned(v, eb) || !aligned(g, eb) || !aligned(beta, eb) || !aligned(y, eb) ||
        !aligned(delta_log, eb) || !aligned(g_log, eb) || !aligned(mask, 4))
        return fail(GDN_ERR_MISALIGNED, "%s: a tensor is not aligned to its element size", fn);
    if (state_in != state_out && overlap(state_in, s_b, state_out, s_b))
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: state_out overlaps state_in without being the same buffer", fn);

    if (take_forced_failure()) return forced_failure(fn);
    cudaError_t e;
    const int sms = current_sm_count(&e);
    if (e != cudaSuccess) return cuda_fail(fn, "device query", e);
    const gdn::Geometry geo =
        gdn::record_geometry((int)Dk, B * Hv, Dv, T, eb, dtype == GDN_DTYPE_BF16, sms);
    if ((B * Hv) > (int64_t)INT32_MAX / geo.row_blocks)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: grid too large (B*Hv*row_blocks > 2^31-1)", fn);
    gdn::RecordArgs a{q, k, v, g, beta, state_in, mask, y, state_out, delta_log, k_log, g_log,
                      B, T, Hk, Hv, Dv, geo.rows_cta, geo.row_blocks, geo.tc,
                      aligned(v, 16) && (Dv * eb) % 16 == 0, mapping == GDN_GQA_TILED,
                      tstate && dtype != GDN_DTYPE_F32};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((geo.mma || T >= gdn::kTcMinSteps) && gdn::record_tc_eligible(a, (int)Dk, dtype == GDN_DTYPE_BF16)) {
        e = gdn::launch_record_tc(a, sms, s);  // one chunk on tcgen05, the TMA-fed stream
    } else {
        switch (dtype) {
        case GDN_DTYPE_F32: e = gdn::launch_record_f32((int)Dk, a, geo, s); break;
        case GDN_DTYPE_BF16: e = gdn::launch_record_bf16((int)Dk, a, geo, s); break;
        case GDN_DTYPE_F16: e = gdn::launch_record_f16((int)Dk, a, geo, s); break;
        }
    }
    if (e != cudaSuccess) return cuda_fail(fn, "launch", e);
    return ok();
}

gdn_status replay_impl(const char *fn, const void *delta_log, const void *k_log, const void *g_log,
                       const void *state_in, const uint32_t *mask, void *state_out, int64_t B,
                       int64_t T, int64_t Hv, int64_t Dk, int64_t Dv, int64_t accepted,
                       const int32_t *accepted_per_seq, gdn_dtype dtype, bool tstate,
                       gdn_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(GDN_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dtype);
    if (B <= 0 || T <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: B, T, Hv, Dk, Dv must all be > 0 (got %lld %lld %lld %lld %lld)", fn,
                    (long long)B, (long long)T, (long long)Hv, (long long)Dk, (long long)Dv);
    if (accepted < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: accepted (%lld) must be >= 0", fn,
                    (long long)accepted);
    if (!delta_log || !k_log || !g_log || !state_in || !state_out)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: delta_log, k_log, g_log, state_in, state_out must be non-NULL", fn);
    if (Dk % 32 != 0 || !gdn::supported_dk(Dk))
        return fail(GDN_ERR_UNSUPPORTED, "%s: Dk = %lld not supported (32, 64, 128, 192, 256)", fn,
                    (long long)Dk);
    const int64_t d_b = nbytes({B, T, Hv, Dv}, eb), kl_b = nbytes({B, T, Hv, Dk}, eb);
    const int64_t s_b = nbytes({B, Hv, Dv, Dk}, tstate ? eb : 4), g_b = nbytes({B, T, Hv}, eb);
    const int64_t m_b = nbytes({B, T}, 4);
    if (d_b < 0 || kl_b < 0 || s_b < 0 || g_b < 0 || m_b < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: tensor sizes overflow int64", fn);
    if (!aligned(k_log, 16) || !aligned(state_in, 16) || !aligned(state_out, 16))
        return fail(GDN_ERR_MISALIGNED, "%s: k_log, state_in, state_out must be 16-byte aligned", fn);
    if (!aligned(delta_log, eb) || !aligned(g_log, eb) || !aligned(mask, 4) ||
        !aligned(accepted_per_seq, 4))
        return fail(GDN_ERR_MISALIGNED, "%s: a tensor is not aligned to its element size", fn);
    if (state_in != state_out && overlap(state_in, s_b, state_out, s_b))
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: state_out overlaps state_in without being the same buffer", fn);

    const int64_t steps = accepted < T ? accepted : T;
    if (!accepted_per_seq && steps == 0 && state_in == state_out)
        return ok();  // identity, nothing to do
    if (take_forced_failure()) return forced_failure(fn);
    cudaError_t e;
    const int sms = current_sm_count(&e);
    if (e != cudaSuccess) return cuda_fail(fn, "device query", e);
    const gdn::Geometry geo = gdn::replay_geometry((int)Dk, B * Hv, Dv, steps, eb, sms);
    if ((B * Hv) > (int64_t)INT32_MAX / geo.row_blocks)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: grid too large", fn);
    gdn::ReplayArgs a{delta_log, k_log, g_log, state_in, mask, state_out, B, T, Hv, Dv, steps,
                      geo.rows_cta, geo.row_blocks, geo.tc,
                      aligned(delta_log, 16) && (Dv * eb) % 16 == 0, accepted_per_seq,
                      tstate && dtype != GDN_DTYPE_F32};
    bool streamed = false;
    e = gdn::launch_replay_stream(static_cast<gdn::DType>(dtype), (int)Dk, a, sms,
                                  reinterpret_cast<cudaStream_t>(stream), &streamed);
    if (e == cudaSuccess && !streamed)
        e = gdn::launch_replay(static_cast<gdn::DType>(dtype), (int)Dk, a, geo,
                               reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(fn, "launch", e);
    return ok();
}

gdn_status chunk_prefill_impl(const char *fn, const void *q, const void *k, const void *v,
                              const void *g, const void *beta, const float *state_in,
                              const uint32_t *mask, void *y, float *state_out, void *delta_log,
                              void *k_log, void *g_log, int64_t B, int64_t T, int64_t Hk,
                              int64_t Hv, int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                              void *workspace, size_t workspace_bytes, gdn_dtype dtype,
                              gdn_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(GDN_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dtype);
    if (mapping != GDN_GQA_BLOCK && mapping != GDN_GQA_TILED)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: unknown GQA mapping %d", fn, (int)mapping);
    if (B <= 0 || T <= 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: B, T, Hk, Hv, Dk, Dv must all be > 0 (got %lld %lld %lld %lld %lld %lld)", fn,
                    (long long)B, (long long)T, (long long)Hk, (long long)Hv, (long long)Dk, (long long)Dv);
    if (Hv % Hk != 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: Hv (%lld) must be a multiple of Hk (%lld)", fn,
                    (long long)Hv, (long long)Hk);
    if (!q || !k || !v || !g || !beta || !state_in || !y || !state_out || !workspace)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: q, k, v, g, beta, state_in, y, state_out, workspace must be non-NULL", fn);
    if (Dk % 32 != 0 || !gdn::supported_dk(Dk))
        return fail(GDN_ERR_UNSUPPORTED, "%s: Dk = %lld not supported (32, 64, 128, 192, 256)", fn,
                    (long long)Dk);
    const int64_t qk_b = nbytes({B, T, Hk, Dk}, eb), v_b = nbytes({B, T, Hv, Dv}, eb);
    const int64_t s_b = nbytes({B, Hv, Dv, Dk}, 4), kl_b = nbytes({B, T, Hv, Dk}, eb);
    const int64_t gb_b = nbytes({B, T, Hv}, eb), m_b = nbytes({B, T}, 4);
    const int64_t ws_b = gdn::chunk_workspace_bytes(B, T, Hv);
    if (qk_b < 0 || v_b < 0 || s_b < 0 || kl_b < 0 || gb_b < 0 || m_b < 0 || ws_b < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: tensor sizes overflow int64", fn);
    if (workspace_bytes < (uint64_t)ws_b)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: workspace too small: need %lld bytes, have %llu", fn,
                    (long long)ws_b, (unsigned long long)workspace_bytes);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(state_in, 16) || !aligned(state_out, 16) ||
        !aligned(k_log, 16) || !aligned(workspace, 16))
        return fail(GDN_ERR_MISALIGNED,
                    "%s: q, k, state_in, state_out, k_log, workspace must be 16-byte aligned", fn);
    if (!aligned(v, eb) || !aligned(g, eb) || !aligned(beta, eb) || !aligned(y, eb) ||
        !aligned(delta_log, eb) || !aligned(g_log, eb) || !aligned(mask, 4))
        return fail(GDN_ERR_MISALIGNED, "%s: a tensor is not aligned to its element size", fn);
    if (state_in != state_out && overlap(state_in, s_b, state_out, s_b))
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: state_out overlaps state_in without being the same buffer", fn);

    gdn::ChunkArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
    a.state_in = state_in; a.mask = mask; a.y = y; a.state_out = state_out;
    a.delta_log = delta_log; a.k_log = k_log; a.g_log = g_log;
    a.workspace = static_cast<float *>(workspace);
    a.B = B; a.T = T; a.Hk = Hk; a.Hv = Hv; a.Dv = Dv;
    a.nchunks = ceil_div(T, gdn::kCkC);
    a.row_blocks = ceil_div(Dv, gdn::kCkRows);
    a.vec_v = aligned(v, 16) && (Dv * eb) % 16 == 0;
    a.tiled_gqa = mapping == GDN_GQA_TILED;
    if ((B * Hv) > (int64_t)INT32_MAX / a.nchunks || (B * Hv) > (int64_t)INT32_MAX / a.row_blocks)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: grid too large", fn);
    if (take_forced_failure()) return forced_failure(fn);
    const cudaError_t e = gdn::launch_chunk(static_cast<gdn::DType>(dtype), (int)Dk, a,
                                            reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(fn, "launch", e);
    return ok();
}

gdn_status chunk_replay_impl(const char *fn, const void *delta_log, const void *k_log,
                             const void *g_log, const float *state_in, const uint32_t *mask,
                             float *state_out, int64_t B, int64_t T, int64_t Hv, int64_t Dk,
                             int64_t Dv, int64_t accepted, const int32_t *accepted_per_seq,
                             void *workspace, size_t workspace_bytes, gdn_dtype dtype,
                             gdn_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(GDN_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dtype);
    if (B <= 0 || T <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: B, T, Hv, Dk, Dv must all be > 0 (got %lld %lld %lld %lld %lld)", fn,
                    (long long)B, (long long)T, (long long)Hv, (long long)Dk, (long long)Dv);
    if (accepted < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: accepted (%lld) must be >= 0", fn, (long long)accepted);
    if (!delta_log || !k_log || !g_log || !state_in || !state_out || !workspace)
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: delta_log, k_log, g_log, state_in, state_out, workspace must be non-NULL", fn);
    if (Dk % 32 != 0 || !gdn::supported_dk(Dk))
        return fail(GDN_ERR_UNSUPPORTED, "%s: Dk = %lld not supported (32, 64, 128, 192, 256)", fn,
                    (long long)Dk);
    const int64_t d_b = nbytes({B, T, Hv, Dv}, eb), kl_b = nbytes({B, T, Hv, Dk}, eb);
    const int64_t s_b = nbytes({B, Hv, Dv, Dk}, 4), g_b = nbytes({B, T, Hv}, eb);
    const gdn::ReplayTcPlan plan = gdn::replay_tc_plan(B, T, Hv, Dk, Dv);
    if (d_b < 0 || kl_b < 0 || s_b < 0 || g_b < 0 || plan.bytes < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: tensor sizes overflow int64", fn);
    if (workspace_bytes < (uint64_t)plan.bytes)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: workspace too small: need %lld bytes, have %llu", fn,
                    (long long)plan.bytes, (unsigned long long)workspace_bytes);
    if (!aligned(state_in, 16) || !aligned(state_out, 16) || !aligned(workspace, 16))
        return fail(GDN_ERR_MISALIGNED, "%s: state_in, state_out, workspace must be 16-byte aligned", fn);
    if (!aligned(delta_log, eb) || !aligned(k_log, eb) || !aligned(g_log, eb) || !aligned(mask, 4) ||
        !aligned(accepted_per_seq, 4))
        return fail(GDN_ERR_MISALIGNED, "%s: a tensor is not aligned to its element size", fn);
    if (state_in != state_out && overlap(state_in, s_b, state_out, s_b))
        return fail(GDN_ERR_INVALID_ARGUMENT,
                    "%s: state_out overlaps state_in without being the same buffer", fn);
    const int64_t grid = plan.splits * B * Hv * plan.row_blocks;
    if (grid > (int64_t)INT32_MAX || B * Hv > (int64_t)INT32_MAX)
        return fail(GDN_ERR_INVALID_ARGUMENT, "%s: grid too large", fn);

    if (take_forced_failure()) return forced_failure(fn);
    cudaError_t e;
    const int sms = current_sm_count(&e);
    if (e != cudaSuccess) return cuda_fail(fn, "device query", e);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    gdn::ReplayTcArgs a{};
    a.delta_log = delta_log; a.k_log = k_log; a.g_log = g_log;
    a.state_in = state_in; a.mask = mask; a.state_out = state_out;
    a.acc_b = accepted_per_seq;
    a.w = reinterpret_cast<float *>(ws + plan.w_off);
    a.gam = reinterpret_cast<float *>(ws + plan.gam_off);
    a.partial = plan.splits > 1 ? reinterpret_cast<float *>(ws + plan.partial_off) : nullptr;
    a.B = B; a.T = T; a.Hv = Hv; a.Dv = Dv;
    a.steps = accepted_per_seq ? T : (accepted < T ? accepted : T);
    a.row_blocks = plan.row_blocks;
    a.split_steps = plan.split_steps;
    a.splits = plan.splits;
    a.staged = aligned(delta_log, 16) && aligned(k_log, 16) && (Dv * eb) % 16 == 0;
    e = gdn::launch_replay_tc(static_cast<gdn::DType>(dtype), (int)Dk, a,
                              reinterpret_cast<cudaStream_t>(stream), sms);
    if (e != cudaSuccess) return cuda_fail(fn, "launch", e);
    return ok();
}

}  // namespace

extern "C" {

size_t gdn_chunk_replay_workspace_size(int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv) {
    if (B <= 0 || T <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0) return 0;
    const gdn::ReplayTcPlan plan = gdn::replay_tc_plan(B, T, Hv, Dk, Dv);
    return plan.bytes < 0 ? 0 : (size_t)plan.bytes;
}

gdn_status gdn_chunk_replay(const void *delta_log, const void *k_log, const void *g_log,
                            const float *state_in, const uint32_t *mask, float *state_out,
                            int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv,
                            int64_t accepted, const int32_t *accepted_per_seq, void *workspace,
                            size_t workspace_bytes, gdn_dtype dtype, gdn_stream_t stream) {
    return chunk_replay_impl("gdn_chunk_replay", delta_log, k_log, g_log, state_in, mask, state_out,
                             B, T, Hv, Dk, Dv, accepted, accepted_per_seq, workspace,
                             workspace_bytes, dtype, stream);
}

size_t gdn_chunk_prefill_workspace_size(int64_t B, int64_t T, int64_t Hv) {
    if (B <= 0 || T <= 0 || Hv <= 0) return 0;
    const int64_t r = gdn::chunk_workspace_bytes(B, T, Hv);
    return r < 0 ? 0 : (size_t)r;
}

gdn_status gdn_chunk_prefill(const void *q, const void *k, const void *v, const void *g,
                             const void *beta, const float *state_in, const uint32_t *mask,
                             void *y, float *state_out, void *delta_log, void *k_log,
                             void *g_log, int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                             int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping, void *workspace,
                             size_t workspace_bytes, gdn_dtype dtype, gdn_stream_t stream) {
    return chunk_prefill_impl("gdn_chunk_prefill", q, k, v, g, beta, state_in, mask, y, state_out,
                              delta_log, k_log, g_log, B, T, Hk, Hv, Dk, Dv, mapping, workspace,
                              workspace_bytes, dtype, stream);
}

gdn_status gdn_chunk_prefill_noalloc(const void *q, const void *k, const void *v, const void *g,
                                     const void *beta, const float *state_in,
                                     const uint32_t *mask, void *y, float *state_out,
                                     void *delta_log, void *k_log, void *g_log, int64_t B,
                                     int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                                     gdn_gqa_mapping mapping, gdn_dtype dtype,
                                     gdn_stream_t stream) {
    static const char *fn = "gdn_chunk_prefill_noalloc";
    if (B > 0 && T > 0 && Hv > 0) {
        const int64_t need = gdn::chunk_workspace_bytes(B, T, Hv);
        if (need < 0 || (uint64_t)need > gdn::kChunkStaticScratchBytes)
            return fail(GDN_ERR_UNSUPPORTED,
                        "%s: needs %lld bytes of scratch; the library's static scratch holds %llu "
                        "(use gdn_chunk_prefill with a caller workspace)",
                        fn, (long long)need, (unsigned long long)gdn::kChunkStaticScratchBytes);
    }
    float *scratch = nullptr;
    const cudaError_t e = gdn::chunk_static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(fn, "static scratch address", e);
    return chunk_prefill_impl(fn, q, k, v, g, beta, state_in, mask, y, state_out, delta_log,
                              k_log, g_log, B, T, Hk, Hv, Dk, Dv, mapping, scratch,
                              gdn::kChunkStaticScratchBytes, dtype, stream);
}

gdn_status gdn_step_record(const void *q, const void *k, const void *v, const void *g,
                           const void *beta, const float *state_in, const uint32_t *mask,
                           void *y, float *state_out, void *delta_log, void *k_log, void *g_log,
                           int64_t B, int64_t T, int64_t Hk, int64_t Hv, int64_t Dk, int64_t Dv,
                           gdn_dtype dtype, gdn_stream_t stream) {
    return record_impl("gdn_step_record", q, k, v, g, beta, state_in, mask, y, state_out,
                       delta_log, k_log, g_log, B, T, Hk, Hv, Dk, Dv, GDN_GQA_BLOCK, dtype, false,
                       stream);
}

gdn_status gdn_step_record_mapped(const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const float *state_in, const uint32_t *mask,
                                  void *y, float *state_out, void *delta_log, void *k_log,
                                  void *g_log, int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                                  int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                                  gdn_dtype dtype, gdn_stream_t stream) {
    return record_impl("gdn_step_record_mapped", q, k, v, g, beta, state_in, mask, y, state_out,
                       delta_log, k_log, g_log, B, T, Hk, Hv, Dk, Dv, mapping, dtype, false, stream);
}

gdn_status gdn_step_record_tstate(const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const void *state_in, const uint32_t *mask,
                                  void *y, void *state_out, void *delta_log, void *k_log,
                                  void *g_log, int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                                  int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                                  gdn_dtype dtype, gdn_stream_t stream) {
    return record_impl("gdn_step_record_tstate", q, k, v, g, beta, state_in, mask, y, state_out,
                       delta_log, k_log, g_log, B, T, Hk, Hv, Dk, Dv, mapping, dtype, true, stream);
}

gdn_status gdn_state_replay(const void *delta_log, const void *k_log, const void *g_log,
                            const float *state_in, const uint32_t *mask, float *state_out,
                            int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv,
                            int64_t accepted, gdn_dtype dtype, gdn_stream_t stream) {
    return replay_impl("gdn_state_replay", delta_log, k_log, g_log, state_in, mask, state_out, B,
                       T, Hv, Dk, Dv, accepted, nullptr, dtype, false, stream);
}

gdn_status gdn_state_replay_per_seq(const void *delta_log, const void *k_log, const void *g_log,
                                    const float *state_in, const uint32_t *mask,
                                    float *state_out, int64_t B, int64_t T, int64_t Hv,
                                    int64_t Dk, int64_t Dv, const int32_t *accepted,
                                    gdn_dtype dtype, gdn_stream_t stream) {
    if (!accepted)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_state_replay_per_seq: accepted must be non-NULL");
    return replay_impl("gdn_state_replay_per_seq", delta_log, k_log, g_log, state_in, mask,
                       state_out, B, T, Hv, Dk, Dv, T, accepted, dtype, false, stream);
}

gdn_status gdn_state_replay_tstate(const void *delta_log, const void *k_log, const void *g_log,
                                   const void *state_in, const uint32_t *mask, void *state_out,
                                   int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv,
                                   int64_t accepted, const int32_t *accepted_per_seq,
                                   gdn_dtype dtype, gdn_stream_t stream) {
    if (accepted < 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gdn_state_replay_tstate: accepted (%lld) must be >= 0",
                    (long long)accepted);
    return replay_impl("gdn_state_replay_tstate", delta_log, k_log, g_log, state_in, mask,
                       state_out, B, T, Hv, Dk, Dv, accepted_per_seq ? T : accepted,
                       accepted_per_seq, dtype, true, stream);
}

gdn_status gqa_repeat_tiled(const void *src, void *dst, int64_t seq, int64_t hg, int64_t h,
                            int64_t k, gdn_dtype dtype, size_t src_bytes, size_t dst_bytes,
                            gdn_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return fail(GDN_ERR_UNSUPPORTED, "gqa_repeat_tiled: unknown dtype %d", (int)dtype);
    if (seq <= 0 || hg <= 0 || h <= 0 || k <= 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: seq, hg, h, k must all be > 0");
    if (h % hg != 0)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: h (%lld) must be a multiple of hg (%lld)",
                    (long long)h, (long long)hg);
    const int64_t need_src = nbytes({seq, hg, k}, eb);
    if (need_src < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: seq*hg*k overflows");
    const int64_t need_dst = nbytes({seq, h, k}, eb);
    if (need_dst < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: seq*h*k overflows");
    if (!src || !dst) return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: src and dst must be non-NULL");
    if (src_bytes < (uint64_t)need_src)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: src buffer too small: need %lld bytes, have %llu",
                    (long long)need_src, (unsigned long long)src_bytes);
    if (dst_bytes < (uint64_t)need_dst)
        return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: dst buffer too small: need %lld bytes, have %llu",
                    (long long)need_dst, (unsigned long long)dst_bytes);
    if (!aligned(src, eb) || !aligned(dst, eb))
        return fail(GDN_ERR_MISALIGNED, "gqa_repeat_tiled: src / dst not aligned to the element size");
    if (overlap(src, need_src, dst, need_dst))
        return fail(GDN_ERR_INVALID_ARGUMENT, "gqa_repeat_tiled: src and dst overlap");

    if (take_forced_failure()) return forced_failure("gqa_repeat_tiled");
    cudaError_t e;
    const int sms = current_sm_count(&e);
    if (e != cudaSuccess) return cuda_fail("gqa_repeat_tiled", "device query", e);
    gdn::RepeatArgs a;
    a.src = src;
    a.dst = dst;
    a.seq = seq;
    a.hg = hg;
    a.h = h;
    a.row_bytes = k * eb;
    a.elem_bytes = eb;
    a.vec16 = (a.row_bytes % 16 == 0) && aligned(src, 16) && aligned(dst, 16);
    e = gdn::launch_repeat(a, reinterpret_cast<cudaStream_t>(stream), sms);
    if (e != cudaSuccess) return cuda_fail("gqa_repeat_tiled", "launch", e);
    return ok();
}

}  // extern "C"
