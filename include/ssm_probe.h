/* ssm_probe.h -- throughput probes of the B300 SM pipes that bound the selective
 * scan (libssmprobe.so). Measurement only: the scan library does not use it.
 *
 * The selective scan's per-element work (Mamba SSM complete guide, section 5,
 * selective_scan: one exp of dt*A, the products dt*u*B and C*h, the update
 * a*h + b) runs on the SFU (ex2), the FP32 FMA pipe and, for its shared
 * operands, the shared-memory/LSU pipe. These probes measure how much of each
 * one SM delivers per clock, so that the compute roof quoted beside the HBM roof
 * can be reproduced on the machine at hand.
 */
#ifndef SSM_PROBE_H
#define SSM_PROBE_H

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SSM_PROBE_API __attribute__((visibility("default")))
#else
#define SSM_PROBE_API
#endif

/* Runs probe `which` (0..14, listed in pipe_rates.cu: 0 ex2, 1 lg2, 2 rcp, 3 fp32
 * FMA, 4 packed fp32x2 FMA, 5-11 and 13-14 shared-memory load patterns, 12 warp
 * shuffle) on the current device and stream, synchronises the stream, and writes
 * the measured work per clock per SM to *per_clock_per_sm (lanes per clock for
 * the pipes, FP32 FMAs per clock for the packed FMA, warp instructions per clock
 * for the loads and shuffles) and the launch's cycle count to *cycles (nullable).
 * Allocates and frees two small device buffers with cudaMallocAsync on the stream.
 * Returns 0, or a negative code: -1 bad argument, -2 no device, -3 allocation
 * failed, -4 launch or copy failed. */
SSM_PROBE_API int ssm_probe_pipe_rate(int which, double* per_clock_per_sm, double* cycles, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SSM_PROBE_H */
