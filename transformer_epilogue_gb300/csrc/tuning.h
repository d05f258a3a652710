// Launch-shape constants of the shared-memory-staged kernels.  Each can be
// overridden at compile time (-DNAME=value) to measure alternatives; the
// values below are the library's defaults.
#pragma once

// Time limit (ns) handed to each mbarrier test of the staged kernels' waits;
// 0 leaves it to the hardware.
#ifndef EP_MBAR_SUSPEND_NS
#define EP_MBAR_SUSPEND_NS 0
#endif

// 1: every kernel is launched as a programmatic dependent of the preceding
// work in its stream (its launch and prologue overlap that work's tail).
#ifndef EP_PDL
#define EP_PDL 1
#endif

// SkipLayerNormalization: largest tile of rows per stage, shared memory for
// one CTA's stages, minimum resident CTAs per SM the compiler must allow for
// (register cap), and 0/1 to use the staged kernel at all.
#ifndef EP_SLN_TMA_TILE_BYTES
#define EP_SLN_TMA_TILE_BYTES 16384
#endif
#ifndef EP_SLN_TMA_STAGE_BUDGET
#define EP_SLN_TMA_STAGE_BUDGET (64 * 1024)
#endif
#ifndef EP_SLN_TMA_MIN_CTAS
#define EP_SLN_TMA_MIN_CTAS 1
#endif
#ifndef EP_SLN_TMA
#define EP_SLN_TMA 1
#endif
// 1: rows of 16385-32768 elements take the staged kernel with more than 256
// consumer threads where a wide shape covers them exactly (0: the 1024-thread
// register rows).
#ifndef EP_SLN_WIDE
#define EP_SLN_WIDE 1
#endif
// 1: those rows in 16-bit types keep gamma/beta in shared memory when they fit
// beside three stages.
#ifndef EP_SLN_WIDE_PARAMS
#define EP_SLN_WIDE_PARAMS 1
#endif
// 1: 16-bit rows of 18432-30720 elements (multiples of 2048 other than 24576)
// take 4 fragments a thread on H/32 consumer threads (0: 512 threads where
// they cover the row).
#ifndef EP_SLN_WIDE_NV4
#define EP_SLN_WIDE_NV4 1
#endif
// 1: float32 rows of those lengths take 8 fragments a thread on H/32 threads.
#ifndef EP_SLN_WIDE_NV8
#define EP_SLN_WIDE_NV8 1
#endif
// 1: aligned rows of 2 or 3 fragments take one thread a row on the register kernel.
#ifndef EP_SLN_SHORT_REG
#define EP_SLN_SHORT_REG 1
#endif
// 1: one CTA per tile, running CTAs take over the tiles of CTAs they cancel
// (cluster launch control); 0: persistent grid, tiles round-robin.
#ifndef EP_SLN_CLC
#define EP_SLN_CLC 1
#endif

// BiasSoftmax row kernel: the same four, plus the smallest threads-per-row
// the staged kernel may use.
#ifndef EP_SM_TMA_TILE_BYTES
#define EP_SM_TMA_TILE_BYTES 16384
#endif
#ifndef EP_SM_TMA_STAGE_BUDGET
#define EP_SM_TMA_STAGE_BUDGET (64 * 1024)
#endif
#ifndef EP_SM_TMA_MIN_CTAS
#define EP_SM_TMA_MIN_CTAS 1
#endif
#ifndef EP_SM_TMA
#define EP_SM_TMA 1
#endif
// 1: one CTA per tile with cluster launch control; 0: persistent round-robin.
#ifndef EP_SM_CLC
#define EP_SM_CLC 1
#endif
// 1: rows of 16385-32768 columns take the staged row kernel with more than 256
// consumer threads where a wide shape covers them exactly (0: the split-row
// pair).
#ifndef EP_SM_WIDE
#define EP_SM_WIDE 1
#endif
// 1: 16-bit rows of 18432-30720 columns (multiples of 2048) take 4 fragments
// a thread on nfrag/4 consumer threads (0: 512 threads where they cover the row).
#ifndef EP_SM_WIDE_NV4
#define EP_SM_WIDE_NV4 1
#endif
// 1: staged softmax rows of 16-bit types form the exponent with one packed
// fused multiply-add per pair of elements.
// 1: 16-bit rows of 18432-26624 columns take 8 fragments a thread on nfrag/8
// threads, two CTAs an SM (0: nfrag/4 threads of 4 fragments, one CTA).
#ifndef EP_SM_WIDE_2CTA
#define EP_SM_WIDE_2CTA 1
#endif
#ifndef EP_SM_LEAN16
#define EP_SM_LEAN16 1
#endif
// 1: 16-byte-aligned rows of exactly 8 elements take the register kernel's
// one-thread rows; 0: the packed kernel.
#ifndef EP_SM_SHORT_VEC
#define EP_SM_SHORT_VEC 1
#endif
#ifndef EP_SM_TMA_MIN_TPR
#define EP_SM_TMA_MIN_TPR 4
#endif

// Split-row softmax (rows longer than the row kernels hold): bytes of data in
// one stage (4096, 8192 or 16384; the stage also holds as many bytes of bias),
// and shared memory for the stages of one CTA.
// Rows of a window of the split-row pair: their data fills at most this many
// quarters of L2.
#ifndef EP_SM_SPLIT_WINDOW_QUARTERS
#define EP_SM_SPLIT_WINDOW_QUARTERS 3
#endif
#ifndef EP_SM_SPLIT_TILE_BYTES
#define EP_SM_SPLIT_TILE_BYTES 16384
#endif
#ifndef EP_SM_SPLIT_STAGE_BUDGET
#define EP_SM_SPLIT_STAGE_BUDGET (64 * 1024)
#endif

// BiasAdd / QuickGelu: shared memory for one CTA's stages, 0/1 staged kernel.
#ifndef EP_EW_TMA_STAGE_BUDGET
#define EP_EW_TMA_STAGE_BUDGET (64 * 1024)
#endif
#ifndef EP_EW_TMA
#define EP_EW_TMA 1
#endif
#ifndef EP_EW_TMA_MIN_CTAS
#define EP_EW_TMA_MIN_CTAS 1
#endif
// 1: one CTA per tile with cluster launch control; 0: persistent round-robin.
#ifndef EP_EW_CLC
#define EP_EW_CLC 1
#endif
