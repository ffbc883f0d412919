// launch.h -- internal (non-ABI) launch interface between the C ABI in api.cu and
// the kernel translation units. Host code only.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

enum DType { kF32 = 0, kBF16 = 1 };

struct ScanArgs {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    const float* h0;
    void* y;
    float* h_last;
    int64_t batch, dim, seqlen;
    int dstate;
    int softplus;
    int in_dtype, out_dtype;
    bool vec;          // rows of u/delta/z/y/B/C are 16-byte aligned (vector loads allowed)
    // look-back, and the work-balanced time-serial form
    void* workspace;
    size_t workspace_bytes;
    int64_t seg_len;   // time steps per look-back segment (multiple of the chunk)
    int64_t n_seg;
    uint32_t spin_limit;
    int64_t drop_segment;   // test hook: this segment withholds its publication (-1: none)
    // time-serial kernel: 0, or the CTA count of the work-balanced form (the CTAs
    // split the (channel group, chunk) work evenly and pass the state across each
    // split point through `workspace`)
    int64_t bal_ctas;
    // time-serial and look-back kernels, bulk-copy (TMA) path only: walk the
    // sequence from its end (step k reads and writes position seqlen - 1 - k)
    int reverse;
    // directional scans (launch_scan_dir only): traversal order 0 raster, 1 reversed,
    // 2 column-major of a rows x cols image, 3 reversed columns; zoh: exact
    // zero-order-hold input matrix (exp(dt A) - 1) / A * B instead of dt * B
    int order;
    int64_t rows, cols;
    int zoh;
};

struct DecodeArgs {
    float* state;
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    void* y;
    int64_t batch, dim;
    int dstate;
    int softplus;
    int in_dtype, out_dtype;
    bool vec;          // A 16-byte and B, C (4 * element size)-byte aligned: vector loads
    bool tma;          // state, x, delta, z, B, C rows all 16-byte aligned: bulk-copy streaming
};

// Causal depthwise conv1d (+ silu), prefill and single-token update.
struct ConvArgs {
    const void* x;          // prefill (batch, dim, seqlen); update (batch, dim)
    const float* w;         // (dim, width)
    const float* bias;      // (dim) or null
    const float* state_in;  // prefill: (batch, dim, width-1) or null (zeros)
    float* state_out;       // prefill: (batch, dim, width-1) or null; update: the state, in/out
    void* out;              // same shape as x
    int64_t batch, dim, seqlen;
    int width;              // 1..4
    int silu;
    int in_dtype, out_dtype;
    bool vec;               // prefill: x and out rows 16-byte aligned (vector path)
    int64_t seg_len;        // prefill: steps per warp segment (a multiple of conv_block_steps)
    int64_t n_seg;
};

// Backward of the selective scan.
struct BwdArgs {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    const float* h0;
    const void* dout;
    const float* dh_last;
    void* du;               // in_dtype
    void* ddelta;           // in_dtype
    void* dz;               // in_dtype (when z)
    float* dA;              // accumulated (zeroed by the host first)
    float* dB;
    float* dC;
    float* dD;
    float* ddelta_bias;
    float* dh0;
    void* workspace;        // checkpoints, scan_bwd_workspace_bytes
    int64_t batch, dim, seqlen;
    int dstate;
    int softplus;
    int in_dtype, dout_dtype;
    bool vec;               // rows of u/delta/z/dout/du/ddelta/dz 16-byte aligned
};

// Mamba-2 SSD scan (bf16 x, dt, B, C, z; fp32 A, D, dt_bias, states).
struct SsdArgs {
    const void* x;          // (batch, seqlen, nheads, 64)
    const void* dt;         // (batch, seqlen, nheads)
    const float* A;         // (nheads)
    const void* B;          // (batch, seqlen, ngroups, dstate)
    const void* C;
    const float* D;         // (nheads) or null
    const void* z;          // like x, or null
    const float* dt_bias;   // (nheads) or null
    const float* h0;        // (batch, nheads, 64, dstate) or null
    void* y;                // like x, out_dtype
    float* h_last;          // like h0, or null
    int64_t batch, seqlen, nheads, ngroups;
    int dstate;             // 64 or 128
    int softplus;
    int out_dtype;
    // test hooks (0 in every product launch): wait budget of the pipeline waits in
    // mbarrier polls (0: the default), and a withheld compute-side arrival (warp 0
    // skips its first "w o x ready" arrive, so the control warp's wait runs out)
    uint32_t wait_limit;
    int withhold_arrive;
    int64_t drop_ticket;    // test hook: this ticket withholds its state publication (-1: none)
    // work-balanced launch: 0, or the CTA count; the CTAs split the (sequence, chunk)
    // work evenly and pass the state across each split through `workspace` (a
    // 16-byte header with the ticket counter at byte 4, one flag per CTA, one state
    // slot of 64 x dstate floats per CTA), waiting at most spin_limit polls
    void* workspace;
    size_t workspace_bytes;
    int64_t bal_ctas;
    uint32_t spin_limit;
};
__host__ __device__ inline size_t ssd_bal_slots_offset(int64_t ctas) { return 16 + (((size_t)ctas * 4 + 15) / 16) * 16; }
size_t ssd_bal_workspace_bytes(int64_t ctas, int dstate);

// Each returns cudaSuccess or the launch error.
cudaError_t launch_scan_bwd(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_ssd_scan(const SsdArgs& a, cudaStream_t s);
int64_t ssd_chunk_len();
// reads (and optionally clears) the SSD kernel's device status word: 0 or the
// source line of a wait that ran out of budget; synchronises the stream
cudaError_t ssd_status(int* line, bool clear, cudaStream_t s);
// the same for the prefill kernels' bulk-copy waits (kernels_serial.cu)
cudaError_t prefill_status(int* line, bool clear, cudaStream_t s);
size_t scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate);
cudaError_t launch_causal_conv1d(const ConvArgs& a, cudaStream_t s);
cudaError_t launch_conv_update(const ConvArgs& a, cudaStream_t s);
// steps one warp covers per block of the prefill conv (32 16-byte vectors)
int conv_block_steps(int in_dtype);
cudaError_t launch_state_update(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_scan_warp(const ScanArgs& a, cudaStream_t s);
cudaError_t launch_scan_dir(const ScanArgs& a, cudaStream_t s);
// transposes, for each of n (1 .. 3) tensors of the same shape, `images` row-major
// rows x cols images of esize-byte elements (2 or 4) from src[t] into dst[t] (each
// becomes cols x rows), in one launch
cudaError_t launch_transpose_images(const void* const* src, void* const* dst, int n, int64_t images, int64_t rows,
                                    int64_t cols, int esize, cudaStream_t s);
cudaError_t launch_scan_serial_lookback(const ScanArgs& a, int lanes_per_channel, cudaStream_t s);
// channels one CTA of the look-back kernel covers (its segments are planned with it)
int lookback_channels_per_cta(int dstate, int lanes_per_channel, int in_dtype);
cudaError_t launch_scan_thread(const ScanArgs& a, int lanes_per_channel, cudaStream_t s);
cudaError_t launch_scan_scalar(const ScanArgs& a, cudaStream_t s);
// the d_state = 1 kernel's device status word: 0 or the line of a bulk-copy wait
// that ran out of budget (synchronises the stream)
cudaError_t scalar_status(int* line, bool clear, cudaStream_t s);

// Look-back residency: the look-back kernel's launch bounds guarantee this many CTAs
// per SM and the host plans its segments so that every CTA is resident at once
// (a build option).
#ifndef SSM_LB_CTAS_PER_SM
#define SSM_LB_CTAS_PER_SM 3
#endif
constexpr int kLookbackCtasPerSM = SSM_LB_CTAS_PER_SM;

// Look-back workspace geometry (bytes), shared by api.cu and the look-back kernel
// (kernels_serial.cu): a 16-byte header and one descriptor of 16*dstate bytes per
// (channel, segment).
constexpr int kWarpScanItems = 8;                    // time steps per lane per chunk
constexpr int kWarpScanChunk = 32 * kWarpScanItems;  // time steps per warp chunk
size_t lookback_workspace_bytes(int64_t batch, int64_t dim, int dstate, int64_t n_seg);
// Work-balanced time-serial scan: channels one CTA holds, and the workspace bytes
// for `ctas` CTAs (a 16-byte header with the ticket counter, one flag per CTA, one
// state slot of channels x dstate floats per CTA).
int serial_channels_per_cta(int dstate, int lanes_per_channel);
size_t serial_bal_workspace_bytes(int64_t ctas, int dstate, int lanes_per_channel);
// byte offset of the flags and of the state slots in that workspace
constexpr size_t kSerialBalFlags = 16;
__host__ __device__ inline size_t serial_bal_slots_offset(int64_t ctas) { return kSerialBalFlags + (((size_t)ctas * 4 + 15) / 16) * 16; }

}  // namespace ssm
