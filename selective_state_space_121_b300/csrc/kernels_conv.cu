// kernels_conv.cu -- the causal depthwise conv1d + silu that feeds the scan, and its
// single-token decode update.
//
// What is computed (Mamba SSM complete guide (youngju.dev), section 5, "complete
// Mamba implementation": MambaBlock.__init__ builds a depthwise nn.Conv1d with
// kernel d_conv and padding d_conv - 1, forward keeps the first seqlen outputs and
// applies silu before the SSM). PyTorch's Conv1d is a cross-correlation over the
// input padded on the left, so for width W = d_conv:
//     out[b,d,t] = silu( bias[d] + sum_{k<W} w[d,k] * xp[b,d,t+k] ),
//     xp[t'] = x[t' - (W-1)] for t' >= W-1, else the conv state (the W-1 inputs
//     before this call, oldest first; zeros when none).
// The decode update applies the same sum to (state, x_t) and shifts x_t into the
// state.
//
// Why not fused into the scan's prologue: in the block, x_proj maps the conv
// output u to the scan's delta, B and C, so u has to be in memory before the scan
// starts; the scan reads it like any input. The conv is therefore its own pass,
// HBM-bound: per token*channel it reads the input once and writes u once.
//
// Prefill layout: a warp walks a segment of one (b, d) row in blocks of 32
// 16-byte vectors (256 bf16 or 128 fp32 steps); lane i owns vector i of the
// block, so each load and store instruction moves 512 contiguous bytes. The W-1
// inputs before a lane's vector come from lane i-1 by shuffle; lane 0 takes the
// previous block's last inputs (carried in registers) or, at the segment start,
// reads them from x (or the conv state). The next block is loaded while the
// current one computes. Rows are cut into segments only when there are too few
// rows to fill the GPU.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

// V consecutive inputs at row[t ..] widened to fp32; zero past L.
template <typename T, bool kVec>
__device__ __forceinline__ void load_v(const T* row, int64_t t, int64_t L, float* out) {
    constexpr int V = Vec16<T>::kN;
    if (kVec && t + V <= L) {
        Vec16<T>::load(row + t, out);
        return;
    }
#pragma unroll
    for (int k = 0; k < V; k++) out[k] = (t + k < L) ? to_f32(row[t + k]) : 0.f;
}

// V outputs at row[t ..], those before te only.
template <typename Tout, int V, bool kVec>
__device__ __forceinline__ void store_v(Tout* row, int64_t t, int64_t te, const float* v) {
    if (kVec && t + V <= te) {
        if constexpr (sizeof(Tout) == 2 && V == 8) {
            Vec16<Tout>::store(row + t, v);
            return;
        } else if constexpr (sizeof(Tout) == 4) {
#pragma unroll
            for (int k = 0; k < V; k += 4) Vec16<Tout>::store(row + t + k, v + k);
            return;
        } else {   // bf16 out, fp32 in: 4 values, 8 bytes
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
            *reinterpret_cast<uint2*>(row + t) =
                make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
            return;
        }
    }
#pragma unroll
    for (int k = 0; k < V; k++)
        if (t + k < te) row[t + k] = from_f32<Tout>(v[k]);
}

// the padded input at time tau < 0 or tau >= 0 of one row: x itself, else the state
template <typename Tin>
__device__ __forceinline__ float padded(const Tin* xr, const float* st, int hw, int64_t tau) {
    if (tau >= 0) return to_f32(xr[tau]);
    return st ? st[hw + tau] : 0.f;
}

template <typename Tin, typename Tout, int W, bool kVec>
__global__ void __launch_bounds__(kThreads) causal_conv1d_kernel(ConvArgs a) {
    constexpr bool kAcc = sizeof(Tin) == 4;
    constexpr int V = Vec16<Tin>::kN;
    constexpr int HW = W - 1;            // halo width
    constexpr int HA = HW > 0 ? HW : 1;  // array size
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t rows = a.batch * a.dim;
    if (gw >= rows * a.n_seg) return;    // whole warp
    const int64_t row = gw / a.n_seg, seg = gw % a.n_seg;
    const int64_t d = row % a.dim, L = a.seqlen;
    const int64_t tb = seg * a.seg_len, te = min(L, tb + a.seg_len);
    const Tin* xr = static_cast<const Tin*>(a.x) + row * L;
    Tout* orow = static_cast<Tout*>(a.out) + row * L;
    const float* st_in = a.state_in ? a.state_in + row * HW : nullptr;
    float w[W];
#pragma unroll
    for (int k = 0; k < W; k++) w[k] = a.w[d * W + k];
    const float bias = a.bias ? a.bias[d] : 0.f;

    // inputs before the segment (every lane holds them; lane 0 uses them)
    float h[HA];
#pragma unroll
    for (int j = 0; j < HW; j++) h[j] = padded(xr, st_in, HW, tb - HW + j);
    // the state a following call continues from: the last W-1 padded inputs,
    // written by the segment-0 warp after it has read the incoming state (so the
    // two may be the same array)
    __syncwarp();
    if (seg == 0 && a.state_out && lane == 0) {
        float so[HA];
#pragma unroll
        for (int j = 0; j < HW; j++) so[j] = padded(xr, st_in, HW, L - HW + j);
#pragma unroll
        for (int j = 0; j < HW; j++) a.state_out[row * HW + j] = so[j];
    }

    float nv[V];
    if (tb < te) load_v<Tin, kVec>(xr, tb + (int64_t)lane * V, L, nv);
    for (int64_t blk = tb; blk < te; blk += 32 * V) {
        const int64_t t = blk + (int64_t)lane * V;
        float v[V];
#pragma unroll
        for (int k = 0; k < V; k++) v[k] = nv[k];
        if (blk + 32 * V < te) load_v<Tin, kVec>(xr, t + 32 * V, L, nv);
        // the W-1 inputs before this lane's vector
        float prev[HA];
#pragma unroll
        for (int j = 0; j < HW; j++) {
            const float up = __shfl_up_sync(0xffffffffu, v[V - HW + j], 1);
            prev[j] = lane == 0 ? h[j] : up;
        }
#pragma unroll
        for (int j = 0; j < HW; j++) h[j] = __shfl_sync(0xffffffffu, v[V - HW + j], 31);
        float o[V];
#pragma unroll
        for (int k = 0; k < V; k++) {
            float acc = bias;
#pragma unroll
            for (int i = 0; i < W; i++) {
                const int e = k + i;   // index into prev ++ v
                acc = fmaf(w[i], e < HW ? prev[e] : v[e - HW], acc);
            }
            o[k] = a.silu ? silu_acc<kAcc>(acc) : acc;
        }
        if (t < te) store_v<Tout, V, kVec>(orow, t, te, o);
    }
}

// One decode token per (b, d) thread: the state row (W-1 fp32 inputs, oldest
// first) and x give the output; the state drops its oldest entry and takes x.
template <typename Tin, typename Tout, int W>
__global__ void __launch_bounds__(256) conv_update_kernel(ConvArgs a) {
    constexpr bool kAcc = sizeof(Tin) == 4;
    constexpr int HW = W - 1;
    constexpr int HA = HW > 0 ? HW : 1;
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= a.batch * a.dim) return;
    const int64_t d = i % a.dim;
    float* st = a.state_out + i * HW;
    float s[HA];
#pragma unroll
    for (int j = 0; j < HW; j++) s[j] = st[j];
    const float xt = to_f32(static_cast<const Tin*>(a.x)[i]);
    float acc = a.bias ? a.bias[d] : 0.f;
#pragma unroll
    for (int j = 0; j < HW; j++) acc = fmaf(a.w[d * W + j], s[j], acc);
    acc = fmaf(a.w[d * W + HW], xt, acc);
    static_cast<Tout*>(a.out)[i] = from_f32<Tout>(a.silu ? silu_acc<kAcc>(acc) : acc);
#pragma unroll
    for (int j = 0; j + 1 < HW; j++) st[j] = s[j + 1];
    if constexpr (HW > 0) st[HW - 1] = xt;
}

template <typename Tin, typename Tout, int W>
cudaError_t launch_fwd(const ConvArgs& a, cudaStream_t s) {
    const int64_t warps = a.batch * a.dim * a.n_seg;
    if (warps == 0) return cudaSuccess;
    const int64_t ctas = (warps + kWarps - 1) / kWarps;
    if (ctas > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
    if (a.vec) causal_conv1d_kernel<Tin, Tout, W, true><<<(unsigned)ctas, kThreads, 0, s>>>(a);
    else causal_conv1d_kernel<Tin, Tout, W, false><<<(unsigned)ctas, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int W>
cudaError_t launch_upd(const ConvArgs& a, cudaStream_t s) {
    const int64_t n = a.batch * a.dim;
    if (n == 0) return cudaSuccess;
    conv_update_kernel<Tin, Tout, W><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t by_width(const ConvArgs& a, bool update, cudaStream_t s) {
    switch (a.width) {
        case 1: return update ? launch_upd<Tin, Tout, 1>(a, s) : launch_fwd<Tin, Tout, 1>(a, s);
        case 2: return update ? launch_upd<Tin, Tout, 2>(a, s) : launch_fwd<Tin, Tout, 2>(a, s);
        case 3: return update ? launch_upd<Tin, Tout, 3>(a, s) : launch_fwd<Tin, Tout, 3>(a, s);
        default: return update ? launch_upd<Tin, Tout, 4>(a, s) : launch_fwd<Tin, Tout, 4>(a, s);
    }
}

cudaError_t dispatch(const ConvArgs& a, bool update, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? by_width<__nv_bfloat16, __nv_bfloat16>(a, update, s)
                                    : by_width<__nv_bfloat16, float>(a, update, s);
    return a.out_dtype == kBF16 ? by_width<float, __nv_bfloat16>(a, update, s) : by_width<float, float>(a, update, s);
}

}  // namespace

int conv_block_steps(int in_dtype) { return 32 * (in_dtype == kBF16 ? 8 : 4); }

cudaError_t launch_causal_conv1d(const ConvArgs& a, cudaStream_t s) { return dispatch(a, false, s); }
cudaError_t launch_conv_update(const ConvArgs& a, cudaStream_t s) { return dispatch(a, true, s); }

}  // namespace ssm
