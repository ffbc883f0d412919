// api.cu -- the C ABI of libssmscan.so (declared in include/ssm_scan.h): argument
// validation, algorithm choice and launches on the caller's stream. The library
// allocates nothing and never synchronises except in ssm_query_status.
#include <string.h>

#include <algorithm>

#include "launch.h"
#include "ssm_scan.h"

namespace {

using ssm::DecodeArgs;
using ssm::BwdArgs;
using ssm::ConvArgs;
using ssm::SsdArgs;
using ssm::ScanArgs;

constexpr uint32_t kSpinLimit = 1u << 20;   // look-back waits: ~0.1-1 s before giving up
constexpr int64_t kSMs = 148;               // B300
// CTAs per SM the work-balanced time-serial form may use (its workspace is sized
// for this many; the launch uses the kernel's actual occupancy, if smaller)
constexpr int64_t kSerialBalCtasPerSM = 8;
// CTAs per SM the work-balanced SSD launch may use (its workspace is sized for this many)
constexpr int64_t kSsdBalCtasPerSM = 2;
// look-back geometry (build options): CTAs per SM aimed at, shortest segment.
// Measured with 2048 against 256 steps (the look-back chooses the segment count
// to fill the SMs; the minimum binds only on shorter sequences): (8, 192, 3136, 16)
// 276 -> 80 us (the warp scan took 112), (1, 1536, 16384, 16) 372 -> 269 us,
// (8, 384, 784, 16) 74 -> 61 us (warp scan 65); the long (1, 1536, 131072, 16)
// workload's segments are longer than either.
#ifndef SSM_LB_MIN_SEG
#define SSM_LB_MIN_SEG 256
#endif
constexpr int64_t kLookbackCtasPerSM = ssm::kLookbackCtasPerSM;
constexpr int64_t kLookbackMinSeg = SSM_LB_MIN_SEG;
// lanes per channel of the time-serial kernel at dstate >= 4 (a build option; 2 is
// also built for dstate 16)
#ifndef SSM_SERIAL_LANES
#define SSM_SERIAL_LANES 4
#endif
constexpr int kSerialLanes = SSM_SERIAL_LANES;
// channels from which the time-serial kernels have >= ~4 warps per SM (4 lanes per
// channel at dstate >= 4; 8 lanes per channel at dstate 1)
constexpr int64_t kSerialMinChannels = kSMs * 32;

size_t esize(int dtype) { return dtype == SSM_BF16 ? 2 : 4; }

bool valid_dtype(int dt) { return dt == SSM_F32 || dt == SSM_BF16; }

bool valid_n(int64_t n) { return n == 1 || n == 2 || n == 4 || n == 8 || n == 16; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// product of non-negative sizes, -1 on overflow past 2^62
int64_t mul(int64_t a, int64_t b) {
    if (a < 0 || b < 0) return -1;
    if (a == 0 || b == 0) return 0;
    if (a > ((int64_t)1 << 62) / b) return -1;
    return a * b;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

struct Plan {
    int algo;
    int64_t n_seg, seg_len;
    int lanes_per_channel;
};

// Channels are the unit of parallel work for the serial-carry algorithms; the
// look-back cuts time into segments when there are too few channels to fill the
// B300's 148 SMs.
// Segments of the serial look-back: one CTA per (channel group, segment); at most
// kLookbackCtasPerSM CTAs per SM in all (one wave), segments a multiple of 256
// steps (a whole number of chunks) and at least kLookbackMinSeg steps long.
void plan_lookback(Plan& p, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype) {
    const int G = dstate >= 4 ? kSerialLanes : (int)dstate;
    p.lanes_per_channel = G;
    const int64_t ch_per_cta = ssm::lookback_channels_per_cta((int)dstate, G, in_dtype);
    const int64_t groups = dim > 0 ? (dim + ch_per_cta - 1) / ch_per_cta : 1;
    const int64_t ctas_per_seg = groups * (batch > 0 ? batch : 1);
    // all CTAs resident at once (the kernel's launch bounds guarantee
    // kLookbackCtasPerSM per SM): a CTA that starts only when a first-wave CTA
    // leaves runs its segment after the whole first wave -- at (1, 1536, 131072, 16)
    // rounding up to 19 segments (456 CTAs for 444 slots) cost 60%
    const int64_t target_ctas = kSMs * kLookbackCtasPerSM;
    int64_t want = target_ctas / ctas_per_seg;
    if (want < 1) want = 1;
    const int64_t gran = ssm::kWarpScanChunk;
    int64_t seg_len = (seqlen + want - 1) / want;
    seg_len = ((seg_len + gran - 1) / gran) * gran;
    if (seg_len < kLookbackMinSeg) seg_len = kLookbackMinSeg;
    p.seg_len = seg_len;
    p.n_seg = seqlen > 0 ? (seqlen + seg_len - 1) / seg_len : 1;
}

Plan plan_scan(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int algo, int in_dtype) {
    Plan p{algo, 1, seqlen, 1};
    const int64_t channels = batch * dim;
    if (p.algo == SSM_ALGO_AUTO) {
        // Time-serial lanes when the channels alone fill the GPU (the fewest
        // instructions per element); otherwise split time: across CTAs (the
        // look-back) when that yields at least one CTA per SM, else across a
        // warp's lanes. Measured at (1, 1536, 131072, 16): look-back 2.3 ms,
        // warp scan 6.9 ms.
        if (channels >= kSerialMinChannels) {
            p.algo = SSM_ALGO_THREAD;
        } else {
            p.algo = SSM_ALGO_WARPSCAN;
            if (channels > 0) {
                Plan lb{SSM_ALGO_LOOKBACK, 1, seqlen, 1};
                plan_lookback(lb, batch, dim, seqlen, dstate, in_dtype);
                const int G = dstate >= 4 ? kSerialLanes : (int)dstate;
                const int64_t ch_per_cta = ssm::lookback_channels_per_cta((int)dstate, G, in_dtype);
                const int64_t ctas = lb.n_seg * ((dim + ch_per_cta - 1) / ch_per_cta) * batch;
                if (lb.n_seg > 1 && ctas >= kSMs) p.algo = SSM_ALGO_LOOKBACK;
            }
        }
    }
    if (p.algo == SSM_ALGO_THREAD) p.lanes_per_channel = dstate >= 4 ? kSerialLanes : (int)dstate;
    if (p.algo == SSM_ALGO_LOOKBACK) plan_lookback(p, batch, dim, seqlen, dstate, in_dtype);
    return p;
}

size_t workspace_for(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int algo, int in_dtype) {
    Plan p = plan_scan(batch, dim, seqlen, dstate, algo, in_dtype);
    if (p.algo == SSM_ALGO_THREAD && dstate > 1) {
        // the work-balanced time-serial form: at most one CTA per channel group and
        // kSerialBalCtasPerSM per SM
        const int64_t cpc = ssm::serial_channels_per_cta((int)dstate, p.lanes_per_channel);
        const int64_t units = ((dim + cpc - 1) / cpc) * batch;
        const int64_t ctas = std::min<int64_t>(units, kSMs * kSerialBalCtasPerSM);
        return std::max<size_t>(16, ssm::serial_bal_workspace_bytes(ctas, (int)dstate, p.lanes_per_channel));
    }
    if (p.algo != SSM_ALGO_LOOKBACK) return 16;
    return ssm::lookback_workspace_bytes(batch, dim, (int)dstate, p.n_seg);
}

// Workspace of the column-order directional walks: the scan's own part (`inner`
// bytes), then transposed copies of u, delta, (z), B, C and y, each 256-byte aligned.
struct DirScratch {
    size_t inner, u, d, z, B, C, y, total;
};
size_t round256(size_t v) { return (v + 255) / 256 * 256; }
DirScratch dir_scratch(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype, int out_dtype,
                       bool has_z, size_t inner) {
    DirScratch r;
    const size_t nx = (size_t)batch * (size_t)dim * (size_t)seqlen, nbc = (size_t)batch * (size_t)dstate * seqlen;
    const size_t ei = esize(in_dtype), eo = esize(out_dtype);
    r.inner = round256(inner);
    r.u = r.inner;
    r.d = r.u + round256(nx * ei);
    r.z = r.d + round256(nx * ei);
    r.B = r.z + (has_z ? round256(nx * ei) : 0);
    r.C = r.B + round256(nbc * ei);
    r.y = r.C + round256(nbc * ei);
    r.total = r.y + round256(nx * eo);
    return r;
}

int scan_impl(const void* u, const void* delta, const float* A, const void* B, const void* C,
              const float* D, const void* z, const float* delta_bias, int softplus,
              const float* h0, void* y, float* h_last, int64_t batch, int64_t dim,
              int64_t seqlen, int64_t dstate, int in_dtype, int out_dtype, void* workspace,
              size_t workspace_bytes, int algo, void* stream, int64_t drop_segment,
              uint32_t spin_limit, int order = -1, int64_t rows = 0, int64_t cols = 0, int zoh = 0) {
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || seqlen < 0) return SSM_ERR_DIM;
    // directional scans (order >= 0): the traversal must be one of the four and, for
    // the column orders, cover the rows x cols image exactly
    if (order >= 0 && (order > 3 || (order >= 2 && (rows < 1 || cols < 1 || mul(rows, cols) != seqlen))))
        return SSM_ERR_ORDER;
    if (order >= 0 && seqlen >= ((int64_t)1 << 31)) return SSM_ERR_DIM;   // 32-bit traversal positions
    if (!valid_n(dstate)) return SSM_ERR_UNSUPPORTED_N;
    if (algo < SSM_ALGO_AUTO || algo > SSM_ALGO_LOOKBACK) return SSM_ERR_ALGO;
    const int64_t n_rows = mul(batch, dim);
    const int64_t n_x = mul(n_rows, seqlen);
    const int64_t n_bc = mul(mul(batch, dstate), seqlen);
    const int64_t n_h = mul(n_rows, dstate);
    if (n_rows < 0 || n_x < 0 || n_bc < 0 || n_h < 0) return SSM_ERR_DIM;
    if (n_x > 0 && (!u || !delta || !y)) return SSM_ERR_NULL;
    if (n_bc > 0 && (!B || !C)) return SSM_ERR_NULL;
    if (dim > 0 && !A) return SSM_ERR_NULL;
    const size_t ei = esize(in_dtype), eo = esize(out_dtype);
    const void* in_ptrs[] = {u, delta, z, B, C};
    for (const void* p : in_ptrs)
        if (p && !aligned(p, ei)) return SSM_ERR_ALIGN;
    if (y && !aligned(y, eo)) return SSM_ERR_ALIGN;
    const void* f32_ptrs[] = {A, D, delta_bias, h0, h_last};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return SSM_ERR_ALIGN;
    // y must not overlap any input; h_last may be h0 exactly, but overlap nothing else
    const size_t bx = (size_t)n_x * ei, by = (size_t)n_x * eo, bbc = (size_t)n_bc * ei,
                 bh = (size_t)n_h * 4, bA = (size_t)dim * dstate * 4, bd = (size_t)dim * 4;
    if (overlap(y, by, u, bx) || overlap(y, by, delta, bx) || overlap(y, by, z, bx) ||
        overlap(y, by, B, bbc) || overlap(y, by, C, bbc) || overlap(y, by, h0, bh) ||
        overlap(y, by, h_last, bh) || overlap(y, by, A, bA) || overlap(y, by, D, bd) ||
        overlap(y, by, delta_bias, bd))
        return SSM_ERR_ALIAS;
    if (h_last && h0 && h_last != h0 && overlap(h_last, bh, h0, bh)) return SSM_ERR_ALIAS;
    if (h_last && (overlap(h_last, bh, u, bx) || overlap(h_last, bh, delta, bx) ||
                   overlap(h_last, bh, z, bx) || overlap(h_last, bh, B, bbc) ||
                   overlap(h_last, bh, C, bbc) || overlap(h_last, bh, A, bA) ||
                   overlap(h_last, bh, D, bd) || overlap(h_last, bh, delta_bias, bd)))
        return SSM_ERR_ALIAS;

    Plan p = plan_scan(batch, dim, seqlen, dstate, algo, in_dtype);
    ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.h0 = h0; a.y = y; a.h_last = h_last;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.dstate = (int)dstate;
    a.softplus = softplus ? 1 : 0; a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    bool vec = (seqlen * (int64_t)ei) % 16 == 0 && (seqlen * (int64_t)eo) % 16 == 0;
    for (const void* q : in_ptrs) vec = vec && (!q || aligned(q, 16));
    vec = vec && (!y || aligned(y, 16));
    a.vec = vec;
    a.seg_len = p.seg_len; a.n_seg = p.n_seg;
    a.drop_segment = drop_segment;
    a.spin_limit = spin_limit;
    cudaStream_t s = (cudaStream_t)stream;
    // the planned algorithm on arguments `b` with workspace (ws, ws_bytes)
    auto run_plan = [&](ScanArgs& b, void* ws, size_t ws_bytes) -> int {
        if (p.algo == SSM_ALGO_LOOKBACK) {
            const size_t need = ssm::lookback_workspace_bytes(batch, dim, (int)dstate, p.n_seg);
            if (!ws || ws_bytes < need) return SSM_ERR_WORKSPACE;
            if (!aligned(ws, 16)) return SSM_ERR_ALIGN;
            b.workspace = ws;
            if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return SSM_ERR_LAUNCH;
            return ssm::launch_scan_serial_lookback(b, p.lanes_per_channel, s) == cudaSuccess ? SSM_OK
                                                                                           : SSM_ERR_LAUNCH;
        }
        if (p.algo == SSM_ALGO_THREAD) {
            // an optional workspace enables the work-balanced form of the time-serial kernel
            if (ws && aligned(ws, 16)) {
                b.workspace = ws;
                b.workspace_bytes = ws_bytes;
            }
            const cudaError_t e = dstate == 1 ? ssm::launch_scan_scalar(b, s)
                                              : ssm::launch_scan_thread(b, p.lanes_per_channel, s);
            return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
        }
        return ssm::launch_scan_warp(b, s) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
    };
    if (order >= 0) {
        // Without the exact-ZOH input matrix, the directional walks take the prefill's
        // own algorithms when the plan is the time-serial one, or the look-back with
        // the workspace to hold it:
        //  - raster: directly; reversed: directly on the bulk-copy path (bf16 inputs,
        //    16-byte aligned rows, dstate > 1: the kernels mirror each copy);
        //  - columns / reversed columns: the raster / reversed walk of the transposed
        //    image, through transposed copies of u, delta, z, B, C and y placed in the
        //    workspace after the scan's own part (dir_workspace_bytes).
        // Everything else takes the warp scan with its per-step position map.
        const bool prefill_plan =
            p.algo == SSM_ALGO_THREAD ||
            (p.algo == SSM_ALGO_LOOKBACK && workspace && aligned(workspace, 16) &&
             workspace_bytes >= ssm::lookback_workspace_bytes(batch, dim, (int)dstate, p.n_seg));
        const bool rev_order = order == SSM_ORDER_REVERSE || order == SSM_ORDER_COLUMNS_REVERSE;
        const bool col_order = order == SSM_ORDER_COLUMNS || order == SSM_ORDER_COLUMNS_REVERSE;
        const bool big_ok = seqlen < ((int64_t)1 << 31) && dim < ((int64_t)1 << 31);
        // the transposed copies keep L, so their rows are 16-byte aligned when L allows
        const bool vec_t = col_order ? ((seqlen * (int64_t)ei) % 16 == 0 && (seqlen * (int64_t)eo) % 16 == 0) : vec;
        const bool rev_ok = !rev_order || (in_dtype == SSM_BF16 && vec_t && dstate > 1 && big_ok);
        bool direct = !zoh && prefill_plan && rev_ok && !col_order;
        const DirScratch ds = dir_scratch(batch, dim, seqlen, dstate, in_dtype, out_dtype, z != nullptr,
                                          workspace_for(batch, dim, seqlen, dstate, p.algo, in_dtype));
        const bool transposed = !zoh && prefill_plan && rev_ok && col_order && workspace && aligned(workspace, 16) &&
                                workspace_bytes >= ds.total && big_ok && rows <= INT32_MAX && cols <= INT32_MAX;
        if (!direct && !transposed) {
            a.order = order; a.rows = rows; a.cols = cols; a.zoh = zoh ? 1 : 0;
            return ssm::launch_scan_dir(a, s) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
        }
        a.reverse = rev_order ? 1 : 0;
        if (transposed) {
            // image i (rows x cols, raster) -> (cols x rows): the column walk's step k is
            // position k of the transposed image
            char* w = static_cast<char*>(workspace);
            void* uT = w + ds.u; void* dT = w + ds.d; void* zT = z ? w + ds.z : nullptr;
            void* BT = w + ds.B; void* CT = w + ds.C; void* yT = w + ds.y;
            const int64_t xi = batch * dim, bi = batch * dstate;
            const void* xs[3] = {u, delta, z};
            void* xd[3] = {uT, dT, zT};
            const void* bcs[2] = {B, C};
            void* bcd[2] = {BT, CT};
            if (ssm::launch_transpose_images(xs, xd, z ? 3 : 2, xi, rows, cols, (int)ei, s) != cudaSuccess ||
                ssm::launch_transpose_images(bcs, bcd, 2, bi, rows, cols, (int)ei, s) != cudaSuccess)
                return SSM_ERR_LAUNCH;
            ScanArgs b = a;
            b.u = uT; b.delta = dT; b.z = zT; b.B = BT; b.C = CT; b.y = yT;
            b.vec = vec_t;
            const int st = run_plan(b, workspace, ds.inner);
            if (st != SSM_OK) return st;
            const void* ys[1] = {yT};
            void* yd[1] = {y};
            return ssm::launch_transpose_images(ys, yd, 1, xi, cols, rows, (int)eo, s) == cudaSuccess ? SSM_OK
                                                                                                    : SSM_ERR_LAUNCH;
        }
    }
    return run_plan(a, workspace, workspace_bytes);
}

}  // namespace

extern "C" {

int ssm_abi_version(void) { return SSM_SCAN_ABI_VERSION; }

const char* ssm_status_string(int status) {
    switch (status) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_NULL: return "SSM_ERR_NULL: a required pointer is NULL";
        case SSM_ERR_DIM: return "SSM_ERR_DIM: negative or overflowing size";
        case SSM_ERR_DTYPE: return "SSM_ERR_DTYPE: unknown dtype";
        case SSM_ERR_ALIGN: return "SSM_ERR_ALIGN: misaligned pointer";
        case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE: workspace missing or too small";
        case SSM_ERR_LAUNCH: return "SSM_ERR_LAUNCH: CUDA launch failed";
        case SSM_ERR_LOOKBACK_TIMEOUT:
            return "SSM_ERR_LOOKBACK_TIMEOUT: look-back wait exhausted its budget";
        case SSM_ERR_UNSUPPORTED_N: return "SSM_ERR_UNSUPPORTED_N: dstate must be 1, 2, 4, 8 or 16";
        case SSM_ERR_ALIAS: return "SSM_ERR_ALIAS: an output overlaps an input";
        case SSM_ERR_ALGO: return "SSM_ERR_ALGO: unknown algorithm";
        case SSM_ERR_WIDTH: return "SSM_ERR_WIDTH: conv width must be 1, 2, 3 or 4";
        case SSM_ERR_SHAPE:
            return "SSM_ERR_SHAPE: SSD needs headdim 64, dstate 64 or 128 and nheads a multiple of ngroups";
        case SSM_ERR_WAIT_TIMEOUT: return "SSM_ERR_WAIT_TIMEOUT: a tensor-core wait exhausted its budget";
        case SSM_ERR_ORDER:
            return "SSM_ERR_ORDER: traversal order not in 0..3, or rows * cols != seqlen for a column order";
        case SSM_ERR_SCRATCH_LIMIT:
            return "SSM_ERR_SCRATCH_LIMIT: problem needs more scratch than the library's fixed 4 MiB area";
    }
    return "unknown ssm status";
}

size_t ssm_scan_workspace_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate) {
    if (batch < 0 || dim < 0 || seqlen < 0 || !valid_n(dstate)) return 16;
    if (mul(mul(batch, dim), seqlen) < 0) return 16;
    // the largest need over the algorithms and input dtypes (the look-back's
    // segments depend on how many channels one CTA holds, which depends on dtype)
    size_t need = 16;
    for (int dt : {(int)SSM_F32, (int)SSM_BF16})
        for (int algo : {(int)SSM_ALGO_AUTO, (int)SSM_ALGO_THREAD, (int)SSM_ALGO_LOOKBACK}) {
            const size_t w = workspace_for(batch, dim, seqlen, dstate, algo, dt);
            if (w > need) need = w;
        }
    return need;
}

int ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, int softplus,
                 const float* h0, void* y, float* h_last, int64_t batch, int64_t dim,
                 int64_t seqlen, int64_t dstate, int in_dtype, int out_dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus, h0, y, h_last, batch, dim,
                     seqlen, dstate, in_dtype, out_dtype, workspace, workspace_bytes,
                     SSM_ALGO_AUTO, stream, -1, kSpinLimit);
}

int ssm_scan_fwd_algo(const void* u, const void* delta, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias,
                      int softplus, const float* h0, void* y, float* h_last, int64_t batch,
                      int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype, int out_dtype,
                      void* workspace, size_t workspace_bytes, int algo, void* stream) {
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus, h0, y, h_last, batch, dim,
                     seqlen, dstate, in_dtype, out_dtype, workspace, workspace_bytes, algo,
                     stream, -1, kSpinLimit);
}

int ssm_scalar_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                        const void* C, const float* D, const void* z, const float* delta_bias,
                        int softplus, const float* h0, void* y, float* h_last, int64_t batch,
                        int64_t dim, int64_t seqlen, int in_dtype, int out_dtype,
                        void* workspace, size_t workspace_bytes, void* stream) {
    // (dim) A, (batch, seqlen) B/C and (batch, dim) h0/h_last are exactly the
    // dstate == 1 layouts of the general entry point
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus, h0, y, h_last, batch, dim,
                     seqlen, 1, in_dtype, out_dtype, workspace, workspace_bytes, SSM_ALGO_AUTO,
                     stream, -1, kSpinLimit);
}

int ssm_test_lookback_timeout(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, void* y, int64_t batch, int64_t dim,
                              int64_t seqlen, int64_t dstate, int in_dtype, void* workspace,
                              size_t workspace_bytes, int64_t drop_segment,
                              uint32_t spin_limit, void* stream) {
    return scan_impl(u, delta, A, B, C, nullptr, nullptr, nullptr, 1, nullptr, y, nullptr, batch,
                     dim, seqlen, dstate, in_dtype, in_dtype, workspace, workspace_bytes,
                     SSM_ALGO_LOOKBACK, stream, drop_segment, spin_limit);
}

int ssm_state_update(float* state, const void* x, const void* delta, const float* A,
                     const void* B, const void* C, const float* D, const void* z,
                     const float* delta_bias, int softplus, void* y, int64_t batch, int64_t dim,
                     int64_t dstate, int in_dtype, int out_dtype, void* stream) {
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0) return SSM_ERR_DIM;
    if (!valid_n(dstate)) return SSM_ERR_UNSUPPORTED_N;
    const int64_t n_rows = mul(batch, dim);
    const int64_t n_h = mul(n_rows, dstate);
    const int64_t n_bc = mul(batch, dstate);
    if (n_rows < 0 || n_h < 0 || n_bc < 0) return SSM_ERR_DIM;
    if (n_rows > 0 && (!state || !x || !delta || !y || !B || !C || !A)) return SSM_ERR_NULL;
    const size_t ei = esize(in_dtype), eo = esize(out_dtype);
    const void* in_ptrs[] = {x, delta, z, B, C};
    for (const void* p : in_ptrs)
        if (p && !aligned(p, ei)) return SSM_ERR_ALIGN;
    if (y && !aligned(y, eo)) return SSM_ERR_ALIGN;
    // the state is streamed with 16-byte vector accesses when dstate >= 4
    if (state && !aligned(state, dstate >= 4 ? 16 : 4)) return SSM_ERR_ALIGN;
    const void* f32_ptrs[] = {A, D, delta_bias};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return SSM_ERR_ALIGN;
    const size_t bh = (size_t)n_h * 4, bx = (size_t)n_rows * ei, by = (size_t)n_rows * eo,
                 bbc = (size_t)n_bc * ei, bA = (size_t)dim * dstate * 4, bd = (size_t)dim * 4;
    if (overlap(y, by, state, bh) || overlap(y, by, x, bx) || overlap(y, by, delta, bx) ||
        overlap(y, by, z, bx) || overlap(y, by, B, bbc) || overlap(y, by, C, bbc) ||
        overlap(y, by, A, bA) || overlap(y, by, D, bd) || overlap(y, by, delta_bias, bd))
        return SSM_ERR_ALIAS;
    if (overlap(state, bh, x, bx) || overlap(state, bh, delta, bx) || overlap(state, bh, z, bx) ||
        overlap(state, bh, B, bbc) || overlap(state, bh, C, bbc) || overlap(state, bh, A, bA) ||
        overlap(state, bh, D, bd) || overlap(state, bh, delta_bias, bd))
        return SSM_ERR_ALIAS;
    DecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.state = state; a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.delta_bias = delta_bias; a.y = y; a.batch = batch; a.dim = dim; a.dstate = (int)dstate;
    a.softplus = softplus ? 1 : 0; a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    a.vec = dstate >= 4 && aligned(A, 16) && aligned(B, 4 * ei) && aligned(C, 4 * ei);
    // bulk copies need 16-byte aligned addresses and sizes: the per-row vectors
    // (dim values of x, delta, z; dstate values of B, C) must be whole 16-byte units
    a.tma = dstate >= 8 && a.vec && aligned(state, 16) && aligned(x, 16) && aligned(delta, 16) &&
            (!z || aligned(z, 16)) && aligned(B, 16) && aligned(C, 16) && (dim * (int64_t)ei) % 16 == 0 &&
            (dstate * (int64_t)ei) % 16 == 0;
    return ssm::launch_state_update(a, (cudaStream_t)stream) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_causal_conv1d_fwd(const void* x, const float* weight, const float* bias,
                          const float* conv_state_in, float* conv_state_out, void* out, int64_t batch,
                          int64_t dim, int64_t seqlen, int64_t width, int silu, int in_dtype,
                          int out_dtype, void* stream) {
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || seqlen < 0) return SSM_ERR_DIM;
    if (width < 1 || width > 4) return SSM_ERR_WIDTH;
    const int64_t n_rows = mul(batch, dim);
    const int64_t n_x = mul(n_rows, seqlen);
    const int64_t n_s = mul(n_rows, width - 1);
    if (n_rows < 0 || n_x < 0 || n_s < 0) return SSM_ERR_DIM;
    if (n_x > 0 && (!x || !out)) return SSM_ERR_NULL;
    if (n_rows > 0 && !weight) return SSM_ERR_NULL;
    const size_t ei = esize(in_dtype), eo = esize(out_dtype);
    if ((x && !aligned(x, ei)) || (out && !aligned(out, eo))) return SSM_ERR_ALIGN;
    const void* f32_ptrs[] = {weight, bias, conv_state_in, conv_state_out};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return SSM_ERR_ALIGN;
    const size_t bx = (size_t)n_x * ei, bo = (size_t)n_x * eo, bs = (size_t)n_s * 4,
                 bw = (size_t)dim * width * 4, bb = (size_t)dim * 4;
    // out overlaps no input; the outgoing state may be the incoming one exactly
    if (overlap(out, bo, x, bx) || overlap(out, bo, weight, bw) || overlap(out, bo, bias, bb) ||
        overlap(out, bo, conv_state_in, bs) || overlap(out, bo, conv_state_out, bs))
        return SSM_ERR_ALIAS;
    if (overlap(conv_state_out, bs, x, bx) || overlap(conv_state_out, bs, weight, bw) ||
        overlap(conv_state_out, bs, bias, bb) ||
        (conv_state_out != conv_state_in && overlap(conv_state_out, bs, conv_state_in, bs)))
        return SSM_ERR_ALIAS;
    ConvArgs a;
    memset(&a, 0, sizeof(a));
    a.x = x; a.w = weight; a.bias = bias; a.state_in = conv_state_in; a.state_out = conv_state_out;
    a.out = out; a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.width = (int)width;
    a.silu = silu ? 1 : 0; a.in_dtype = in_dtype; a.out_dtype = out_dtype;
    a.vec = (seqlen * (int64_t)ei) % 16 == 0 && (seqlen * (int64_t)eo) % 16 == 0 && (!x || aligned(x, 16)) &&
            (!out || aligned(out, 16));
    // one warp per row unless that leaves the GPU short of warps (about 48 per SM
    // keep enough loads in flight for HBM): then rows are cut into segments of
    // whole 32-vector blocks
    const int64_t blk = ssm::conv_block_steps(in_dtype);
    const int64_t blocks = (seqlen + blk - 1) / blk;
    int64_t n_seg = n_rows > 0 ? (kSMs * 48 + n_rows - 1) / n_rows : 1;
    if (n_seg > blocks) n_seg = blocks;
    if (n_seg < 1) n_seg = 1;
    a.seg_len = ((blocks + n_seg - 1) / n_seg) * blk;
    a.n_seg = seqlen > 0 ? (seqlen + a.seg_len - 1) / a.seg_len : 1;
    return ssm::launch_causal_conv1d(a, (cudaStream_t)stream) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_causal_conv1d_update(float* conv_state, const void* x, const float* weight, const float* bias,
                             void* out, int64_t batch, int64_t dim, int64_t width, int silu, int in_dtype,
                             int out_dtype, void* stream) {
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0) return SSM_ERR_DIM;
    if (width < 1 || width > 4) return SSM_ERR_WIDTH;
    const int64_t n_rows = mul(batch, dim);
    const int64_t n_s = mul(n_rows, width - 1);
    if (n_rows < 0 || n_s < 0) return SSM_ERR_DIM;
    if (n_rows > 0 && (!x || !out || !weight || (width > 1 && !conv_state))) return SSM_ERR_NULL;
    const size_t ei = esize(in_dtype), eo = esize(out_dtype);
    if ((x && !aligned(x, ei)) || (out && !aligned(out, eo))) return SSM_ERR_ALIGN;
    const void* f32_ptrs[] = {weight, bias, conv_state};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return SSM_ERR_ALIGN;
    const size_t bx = (size_t)n_rows * ei, bo = (size_t)n_rows * eo, bs = (size_t)n_s * 4,
                 bw = (size_t)dim * width * 4, bb = (size_t)dim * 4;
    if (overlap(out, bo, x, bx) || overlap(out, bo, weight, bw) || overlap(out, bo, bias, bb) ||
        overlap(out, bo, conv_state, bs))
        return SSM_ERR_ALIAS;
    if (overlap(conv_state, bs, x, bx) || overlap(conv_state, bs, weight, bw) || overlap(conv_state, bs, bias, bb))
        return SSM_ERR_ALIAS;
    ConvArgs a;
    memset(&a, 0, sizeof(a));
    a.x = x; a.w = weight; a.bias = bias; a.state_out = conv_state; a.out = out;
    a.batch = batch; a.dim = dim; a.width = (int)width; a.silu = silu ? 1 : 0;
    a.in_dtype = in_dtype; a.out_dtype = out_dtype;

    return ssm::launch_conv_update(a, (cudaStream_t)stream) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate) {
    if (batch < 0 || dim < 0 || seqlen < 0 || !valid_n(dstate)) return 0;
    const int64_t n = mul(mul(mul(batch, dim), (seqlen + 7) / 8), dstate);
    if (n < 0) return 0;
    return ssm::scan_bwd_workspace_bytes(batch, dim, seqlen, (int)dstate);
}

int ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, int softplus, const float* h0,
                 const void* dout, const float* dh_last, void* du, void* ddelta, float* dA, float* dB,
                 float* dC, float* dD, void* dz, float* ddelta_bias, float* dh0, int64_t batch, int64_t dim,
                 int64_t seqlen, int64_t dstate, int in_dtype, int dout_dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
    if (!valid_dtype(in_dtype) || !valid_dtype(dout_dtype)) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || seqlen < 0) return SSM_ERR_DIM;
    if (!valid_n(dstate)) return SSM_ERR_UNSUPPORTED_N;
    const int64_t n_rows = mul(batch, dim);
    const int64_t n_x = mul(n_rows, seqlen);
    const int64_t n_bc = mul(mul(batch, dstate), seqlen);
    const int64_t n_h = mul(n_rows, dstate);
    if (n_rows < 0 || n_x < 0 || n_bc < 0 || n_h < 0) return SSM_ERR_DIM;
    if (n_x > 0 && (!u || !delta || !dout || !du || !ddelta || !B || !C || !dB || !dC)) return SSM_ERR_NULL;
    if (dim > 0 && (!A || !dA)) return SSM_ERR_NULL;
    if (n_x > 0 && z && !dz) return SSM_ERR_NULL;
    if (dim > 0 && D && !dD) return SSM_ERR_NULL;
    const size_t ei = esize(in_dtype), eo = esize(dout_dtype);
    const void* in_ptrs[] = {u, delta, z, B, C, du, ddelta, dz};
    for (const void* q : in_ptrs)
        if (q && !aligned(q, ei)) return SSM_ERR_ALIGN;
    if (dout && !aligned(dout, eo)) return SSM_ERR_ALIGN;
    const void* f32_ptrs[] = {A, D, delta_bias, h0, dh_last, dA, dB, dC, dD, ddelta_bias, dh0};
    for (const void* q : f32_ptrs)
        if (q && !aligned(q, 4)) return SSM_ERR_ALIGN;
    // checkpoints are read and written as 16-byte vectors
    if (workspace && !aligned(workspace, 16)) return SSM_ERR_ALIGN;
    const size_t need = ssm::scan_bwd_workspace_bytes(batch, dim, seqlen, (int)dstate);
    if (need > 0 && (!workspace || workspace_bytes < need)) return SSM_ERR_WORKSPACE;
    // outputs overlap no input and no other output
    const size_t bx = (size_t)n_x * ei, bo = (size_t)n_x * eo, bbc = (size_t)n_bc * ei, bbc4 = (size_t)n_bc * 4,
                 bh = (size_t)n_h * 4, bA = (size_t)dim * dstate * 4, bd = (size_t)dim * 4;
    const struct { const void* p; size_t n; } ins[] = {{u, bx}, {delta, bx}, {z, bx}, {B, bbc}, {C, bbc},
                                                        {A, bA}, {D, bd}, {delta_bias, bd}, {h0, bh},
                                                        {dout, bo}, {dh_last, bh}, {workspace, need}};
    const struct { const void* p; size_t n; } outs[] = {{du, bx}, {ddelta, bx}, {dz, bx}, {dA, bA}, {dB, bbc4},
                                                         {dC, bbc4}, {dD, bd}, {ddelta_bias, bd}, {dh0, bh}};
    for (const auto& o : outs) {
        for (const auto& i : ins)
            if (overlap(o.p, o.n, i.p, i.n)) return SSM_ERR_ALIAS;
        for (const auto& o2 : outs)
            if (&o2 != &o && overlap(o.p, o.n, o2.p, o2.n)) return SSM_ERR_ALIAS;
    }
    cudaStream_t s = (cudaStream_t)stream;
    // the accumulated gradients start at zero
    const struct { void* p; size_t n; } acc[] = {{dA, bA}, {dB, bbc4}, {dC, bbc4}, {dD, bd}, {ddelta_bias, bd}};
    for (const auto& z0 : acc)
        if (z0.p && z0.n && cudaMemsetAsync(z0.p, 0, z0.n, s) != cudaSuccess) return SSM_ERR_LAUNCH;
    BwdArgs a;
    memset(&a, 0, sizeof(a));
    a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
    a.h0 = h0; a.dout = dout; a.dh_last = dh_last; a.du = du; a.ddelta = ddelta; a.dz = dz; a.dA = dA;
    a.dB = dB; a.dC = dC; a.dD = dD; a.ddelta_bias = ddelta_bias; a.dh0 = dh0; a.workspace = workspace;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.dstate = (int)dstate; a.softplus = softplus ? 1 : 0;
    a.in_dtype = in_dtype; a.dout_dtype = dout_dtype;
    bool vec = (seqlen * (int64_t)ei) % 16 == 0 && (seqlen * (int64_t)eo) % 16 == 0;
    const void* vec_ptrs[] = {u, delta, z, dout, du, ddelta, dz};
    for (const void* q : vec_ptrs) vec = vec && (!q || aligned(q, 16));
    a.vec = vec;
    return ssm::launch_scan_bwd(a, s) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_query_status(const void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < 16) return SSM_ERR_WORKSPACE;
    int32_t st = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SSM_ERR_LAUNCH;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_LAUNCH;
    return st;
}


}  // extern "C"

// ssm_ssd_scan_fwd with the kernel's test hooks (wait budget, withheld arrival)
static int ssd_impl(const void* x, const void* dt, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int softplus, const float* h0, void* y, float* h_last,
                    int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups, int64_t dstate,
                    int in_dtype, int out_dtype, void* workspace, size_t workspace_bytes, uint32_t wait_limit,
                    int withhold_arrive, void* stream, int64_t drop_ticket = -1) {
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || in_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (batch < 0 || seqlen < 0 || nheads < 0 || ngroups < 0) return SSM_ERR_DIM;
    if (headdim != 64 || (dstate != 64 && dstate != 128)) return SSM_ERR_SHAPE;
    if (nheads > 0 && (ngroups < 1 || nheads % ngroups != 0)) return SSM_ERR_SHAPE;
    const int64_t n_bh = mul(batch, nheads);
    const int64_t n_dt = mul(n_bh, seqlen);
    const int64_t n_x = mul(n_dt, headdim);
    const int64_t n_bc = mul(mul(mul(batch, seqlen), ngroups), dstate);
    const int64_t n_h = mul(mul(n_bh, headdim), dstate);
    if (n_bh < 0 || n_dt < 0 || n_x < 0 || n_bc < 0 || n_h < 0 || n_bh > INT32_MAX) return SSM_ERR_DIM;
    if (n_x > 0 && (!x || !dt || !B || !C || !y)) return SSM_ERR_NULL;
    if (nheads > 0 && !A) return SSM_ERR_NULL;
    const void* v16[] = {x, z, y, B, C};
    for (const void* p : v16)
        if (p && !aligned(p, 16)) return SSM_ERR_ALIGN;
    if (dt && !aligned(dt, 2)) return SSM_ERR_ALIGN;
    const void* f32_ptrs[] = {A, D, dt_bias, h0, h_last};
    for (const void* p : f32_ptrs)
        if (p && !aligned(p, 4)) return SSM_ERR_ALIGN;
    const size_t eo = esize(out_dtype);
    const size_t bx = (size_t)n_x * 2, by = (size_t)n_x * eo, bdt = (size_t)n_dt * 2, bbc = (size_t)n_bc * 2,
                 bh = (size_t)n_h * 4, bp = (size_t)nheads * 4;
    const void* ins[] = {x, z, dt, B, C, A, D, dt_bias, h0};
    const size_t ins_b[] = {bx, bx, bdt, bbc, bbc, bp, bp, bp, bh};
    for (int i = 0; i < 9; i++)
        if (overlap(y, by, ins[i], ins_b[i])) return SSM_ERR_ALIAS;
    for (int i = 0; i < 8; i++)
        if (overlap(h_last, bh, ins[i], ins_b[i])) return SSM_ERR_ALIAS;
    if (overlap(h_last, bh, y, by) || (h_last != h0 && overlap(h_last, bh, h0, bh))) return SSM_ERR_ALIAS;
    if (n_bh == 0) return SSM_OK;
    SsdArgs a;
    memset(&a, 0, sizeof(a));
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias; a.h0 = h0;
    a.y = y; a.h_last = h_last; a.batch = batch; a.seqlen = seqlen; a.nheads = nheads;
    a.ngroups = ngroups; a.dstate = (int)dstate; a.softplus = softplus ? 1 : 0; a.out_dtype = out_dtype;
    a.wait_limit = wait_limit; a.withhold_arrive = withhold_arrive ? 1 : 0;
    if (workspace) {
        if (!aligned(workspace, 16)) return SSM_ERR_ALIGN;
        a.workspace = workspace;
        a.workspace_bytes = workspace_bytes;
    }
    a.spin_limit = wait_limit ? wait_limit : kSpinLimit;
    a.drop_ticket = drop_ticket;
    return ssm::launch_ssd_scan(a, (cudaStream_t)stream) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

extern "C" {

int ssm_ssd_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                     const float* D, const void* z, const float* dt_bias, int softplus, const float* h0,
                     void* y, float* h_last, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                     int64_t ngroups, int64_t dstate, int in_dtype, int out_dtype, void* stream) {
    return ssd_impl(x, dt, A, B, C, D, z, dt_bias, softplus, h0, y, h_last, batch, seqlen, nheads, headdim, ngroups,
                    dstate, in_dtype, out_dtype, nullptr, 0, 0, 0, stream);
}

int ssm_ssd_scan_fwd_ws(const void* x, const void* dt, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* dt_bias, int softplus, const float* h0,
                        void* y, float* h_last, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                        int64_t ngroups, int64_t dstate, int in_dtype, int out_dtype, void* workspace,
                        size_t workspace_bytes, void* stream) {
    return ssd_impl(x, dt, A, B, C, D, z, dt_bias, softplus, h0, y, h_last, batch, seqlen, nheads, headdim, ngroups,
                    dstate, in_dtype, out_dtype, workspace, workspace_bytes, 0, 0, stream);
}

size_t ssm_ssd_workspace_size(int64_t batch, int64_t nheads, int64_t dstate) {
    if (batch < 0 || nheads < 0 || (dstate != 64 && dstate != 128)) return 16;
    const int64_t units = mul(batch, nheads);
    if (units < 0) return 16;
    // at most one CTA per sequence and kSsdBalCtasPerSM per SM
    const int64_t ctas = std::min<int64_t>(units, kSMs * kSsdBalCtasPerSM);
    return std::max<size_t>(16, ssm::ssd_bal_workspace_bytes(ctas, (int)dstate));
}

int ssm_test_ssd_wait_fault(const void* x, const void* dt, const float* A, const void* B, const void* C,
                            void* y, int64_t batch, int64_t seqlen, int64_t nheads, int64_t ngroups, int64_t dstate,
                            int64_t wait_limit, int withhold_arrive, void* workspace, size_t workspace_bytes,
                            int64_t drop_ticket, void* stream) {
    if (wait_limit < 1 || wait_limit > INT32_MAX) return SSM_ERR_DIM;
    return ssd_impl(x, dt, A, B, C, nullptr, nullptr, nullptr, 1, nullptr, y, nullptr, batch, seqlen, nheads, 64,
                    ngroups, dstate, SSM_BF16, SSM_BF16, workspace, workspace_bytes, (uint32_t)wait_limit,
                    withhold_arrive, stream, drop_ticket);
}

int ssm_test_serial_handover_timeout(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                     void* y, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                     int in_dtype, void* workspace, size_t workspace_bytes, int64_t drop_ticket,
                                     uint32_t spin_limit, void* stream) {
    return scan_impl(u, delta, A, B, C, nullptr, nullptr, nullptr, 1, nullptr, y, nullptr, batch, dim, seqlen,
                     dstate, in_dtype, in_dtype, workspace, workspace_bytes, SSM_ALGO_THREAD, stream, drop_ticket,
                     spin_limit);
}

int64_t ssm_ssd_chunk_len(void) { return ssm::ssd_chunk_len(); }

int ssm_device_status(int clear, void* stream) {
    int line = 0, line2 = 0, line3 = 0;
    if (ssm::ssd_status(&line, clear != 0, (cudaStream_t)stream) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (ssm::prefill_status(&line2, clear != 0, (cudaStream_t)stream) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (ssm::scalar_status(&line3, clear != 0, (cudaStream_t)stream) != cudaSuccess) return SSM_ERR_LAUNCH;
    return (line != 0 || line2 != 0 || line3 != 0) ? SSM_ERR_WAIT_TIMEOUT : SSM_OK;
}

int ssm_scan_fwd_dir(const void* u, const void* delta, const float* A, const void* B, const void* C,
                     const float* D, const void* z, const float* delta_bias, int softplus, const float* h0,
                     void* y, float* h_last, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                     int order, int64_t rows, int64_t cols, int zoh, int in_dtype, int out_dtype, void* stream) {
    if (order < 0) return SSM_ERR_ORDER;
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus, h0, y, h_last, batch, dim, seqlen, dstate,
                     in_dtype, out_dtype, nullptr, 0, SSM_ALGO_WARPSCAN, stream, -1, kSpinLimit, order, rows, cols,
                     zoh);
}

size_t ssm_scan_dir_workspace_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype,
                                   int out_dtype) {
    if (batch < 0 || dim < 0 || seqlen < 0 || !valid_n(dstate) || !valid_dtype(in_dtype) ||
        !valid_dtype(out_dtype))
        return 16;
    if (mul(mul(batch, dim), seqlen) < 0) return 16;
    size_t inner = 16;
    for (int algo : {(int)SSM_ALGO_AUTO, (int)SSM_ALGO_THREAD, (int)SSM_ALGO_LOOKBACK})
        inner = std::max(inner, workspace_for(batch, dim, seqlen, dstate, algo, in_dtype));
    return dir_scratch(batch, dim, seqlen, dstate, in_dtype, out_dtype, true, inner).total;
}

int ssm_scan_fwd_dir_ws(const void* u, const void* delta, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, int softplus, const float* h0,
                        void* y, float* h_last, int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                        int order, int64_t rows, int64_t cols, int zoh, int in_dtype, int out_dtype,
                        void* workspace, size_t workspace_bytes, void* stream) {
    if (order < 0) return SSM_ERR_ORDER;
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus, h0, y, h_last, batch, dim, seqlen, dstate,
                     in_dtype, out_dtype, workspace, workspace_bytes, SSM_ALGO_AUTO, stream, -1, kSpinLimit, order,
                     rows, cols, zoh);
}

}  // extern "C"
