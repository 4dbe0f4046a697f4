/*
 * gdn_decode_diag.h -- diagnostics and test hooks of the GDN decode-step
 * library (include/gdn_decode.h). None of these is needed to run a step;
 * they expose the projection plan and a per-phase timeline for tests and
 * profiling, and the debug flags that make a wait run out on purpose.
 *
 * The pages this library follows keep the same kind of instruments beside
 * their launch: per-width compile metadata and per-kernel step profiles
 * (sgl-amd-mono #89, "Speed Tests and Profiling"), and a test that stalls the
 * first wait to check the deadline path (sgl-amd-mono #89, Kernel checks).
 */
#ifndef GDN_DECODE_DIAG_H_
#define GDN_DECODE_DIAG_H_

#include "gdn_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Test hooks (gdn_decode_config.debug_flags). Never set in production. */
#define GDN_DEBUG_SKIP_NORM_PUBLISH 0x1 /* CTA 0 never publishes its norm partials,
                                           so every CTA's first wait runs out */
#define GDN_DEBUG_TIMELINE 0x2          /* record %globaltimer stamps of each CTA's
                                           phases (read with gdn_decode_debug_timeline) */

/* Synchronise `stream` and copy the phase timeline the last step recorded
 * (handle created with GDN_DEBUG_TIMELINE). cta_stamps receives num_ctas x 48
 * uint64 nanosecond stamps: 0 start (after the previous step), 1 norm
 * partials out, 2 norm sums in (rstd known), 3 normed input built in shared
 * memory, 4
 * projection start, 5 projection end, 6 the first recurrence
 * task's projection partials in, 7 end, 8 that task's inputs done, 9 first
 * MMA, 10 last MMA done, 11 first weight tiles issued, 12 x and residual
 * staged, 13 that task's state written; 16+4j+k the j-th task (j < 4) of a
 * CTA with several tasks (k = 0 its inputs in, 1 its state tile in shared
 * memory, 2 state updated, 3 the task's barrier after the update); 32+n the
 * n-th weight tile issued (n < 16); other slots unused.
 * cta_cap is the capacity
 * in elements; *num_ctas receives the grid size. */
gdn_status gdn_decode_debug_timeline(gdn_decode_t* h, void* stream, uint64_t* cta_stamps,
                                     int32_t cta_cap, int32_t* num_ctas);

/* Host-only diagnostics of the stream-K split of the projection work units
 * (no device call) for a grid of num_ctas CTAs. A unit is one 64-column step
 * (k-step) of one 256-row projection tile (tiles: in_proj_qkvz rows first,
 * then in_proj_ba rows); units are ordered by group g = (k-block g / T,
 * tile g % T) of `kblock` k-steps. Fills *engine (the engine the config runs
 * with), unit_begin[num_ctas+1] (CTA c takes units [unit_begin[c],
 * unit_begin[c+1])), seg_slot[num_ctas][16] (partial slot of the i-th group
 * CTA c touches), ks_first[num_ctas] and nb_slots[num_ctas] (CTA c keeps the
 * normed input of k-steps ks_first[c] + j mod ksteps, j < nb_slots[c]),
 * own_mask[num_ctas] (bit j: CTA c owns window slot j, i.e. publishes its
 * norm partial and writes residual_out of that k-step; each k-step has one
 * owner), tile_count[*num_tiles] (partials per tile; capacity tile_cap),
 * *ksteps and *kblock. Errors as for gdn_decode_create. */
gdn_status gdn_decode_plan(const gdn_decode_config* cfg, int32_t num_ctas, int32_t* engine,
                           int32_t* unit_begin, uint8_t* seg_slot, uint16_t* ks_first, uint8_t* nb_slots,
                           uint32_t* own_mask, uint8_t* tile_count, int32_t tile_cap, int32_t* num_tiles,
                           int32_t* ksteps, int32_t* kblock);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DECODE_DIAG_H_ */
