/*
 * kda_profile.h - measurement hooks of the KDA library.
 *
 * Not part of the computation: these calls let a benchmark time each kernel
 * of a forward with CUDA events recorded on the launching stream, between
 * the kernels, with no extra synchronisation.  They have no counterpart on
 * the pages the library follows.
 */
#ifndef KDA_PROFILE_H_
#define KDA_PROFILE_H_

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Number of kernels ("stages") kda_chunk_fwd launches for these arguments,
 * in launch order; fills names[0..min(count, max_names)) with static
 * strings when names is not NULL.  Returns 0 for invalid arguments. */
int32_t kda_chunk_fwd_stages(const kda_fwd_args *args, const char **names, int32_t max_names);

/* kda_chunk_fwd, with events[i] (a cudaEvent_t created by the caller)
 * recorded on the stream just before stage i and events[count] after the
 * last one.  num_events must be at least count + 1 (KDA_ERR_INVALID_ARG
 * otherwise).  Same results and errors as kda_chunk_fwd. */
kda_status kda_chunk_fwd_profiled(const kda_fwd_args *args, kda_stream_t stream,
                                  void *const *events, int32_t num_events);

#ifdef __cplusplus
}
#endif

#endif /* KDA_PROFILE_H_ */
