/*
 * dg tuning and test hooks (companion of dg.h; not needed for normal use).
 *
 * The library picks every tile shape itself (the pages' automatic choice of block size, cluster size
 * and so on: "DeepSeek Open Source Week - Dia 3", technical features). These calls override that
 * choice process-wide, for sweeps and for tests that must reach one particular kernel specialisation.
 * With no knob set, every choice is automatic. Knobs are plain process-wide integers read once per call
 * (atomically, so setting them from one thread while another calls the library is safe, but a call
 * that races with a change may see either value).
 *
 * When the environment variable DG_TUNING is "1" at the time the library is loaded, the variables
 * DG_BN, DG_PAIR, DG_SPLIT, DG_SWAP, DG_GROUP_M and DG_PDL seed the knobs once; otherwise the
 * environment is never read.
 */
#ifndef DG_TUNING_H
#define DG_TUNING_H

#include <stdint.h>

#include "dg.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
    DG_TUNE_BN = 0,       /* tile width (N extent of a tile): used when the layout has that width */
    DG_TUNE_PAIR = 1,     /* 1 = single-CTA tiles, 2 = CTA-pair (256-row) tiles where the layout has them */
    DG_TUNE_SPLIT = 2,    /* split-K cluster size: 1 (off), 2, 4 or 8 (used when K has that many blocks) */
    DG_TUNE_SWAP = 3,     /* few rows (normal GEMM with M <= 128, masked layout with expected_m <= 128):
                             0 = standard kernel, 1 = few-row (decode) kernel with swapped operands */
    DG_TUNE_GROUP_M = 4,  /* tile raster band height, in row blocks (> 0) */
    DG_TUNE_PDL = 5,      /* programmatic dependent launch: 0 = off, 1 = on (the default) */
    DG_TUNE_COUNT = 6
};

#define DG_TUNE_AUTO (-1)

/* Set one knob; DG_TUNE_AUTO restores the automatic choice. DG_INVALID_ARG for an unknown knob. */
dg_status dg_tuning_set(int knob, int value);

/* The knob's current value (DG_TUNE_AUTO when automatic; DG_TUNE_AUTO for an unknown knob). */
int dg_tuning_get(int knob);

/* Every knob back to automatic. */
void dg_tuning_reset(void);

/*
 * Test hook for the failure path. Arms a one-shot fault for the next call that launches the main
 * block-scaled kernel (the normal GEMM with M > 128 and no split, the m-grouped layouts, the weight
 * gradients): that launch bounds every device wait by wait_limit_ns (> 0) instead of the usual second,
 * and its TMA producer leaves its first pipeline stage unfilled. The MMA issuer's wait on that stage
 * then runs out: the kernel records DG_DEVICE_TIMEOUT, drains its in-flight copies and MMAs, frees its
 * tensor memory and returns, with its output unspecified. Nothing faults; dg_device_status() reports
 * the timeout. Product calls never arm it. DG_INVALID_ARG when wait_limit_ns is 0.
 */
dg_status dg_testing_arm_wait_timeout(uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* DG_TUNING_H */
