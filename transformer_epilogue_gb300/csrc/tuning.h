// Launch-shape constants of the shared-memory-staged kernels.  Each can be
// overridden at compile time (-DNAME=value) to measure alternatives; the
// values below are the library's defaults.
#pragma once

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

// BiasSoftmax row kernel: the same four, plus the smallest threads-per-row
// the staged kernel may use.
#ifndef EP_SM_TMA_TILE_BYTES
#define EP_SM_TMA_TILE_BYTES 16384
#endif
#ifndef EP_SM_TMA_STAGE_BUDGET
#define EP_SM_TMA_STAGE_BUDGET (100 * 1024)
#endif
#ifndef EP_SM_TMA_MIN_CTAS
#define EP_SM_TMA_MIN_CTAS 1
#endif
#ifndef EP_SM_TMA
#define EP_SM_TMA 1
#endif
#ifndef EP_SM_TMA_MIN_TPR
#define EP_SM_TMA_MIN_TPR 16
#endif

// Split-row softmax (rows longer than the row kernels hold): shared memory for
// the stages of one CTA (each stage is a 16 KB data chunk + its 16 KB of bias).
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
