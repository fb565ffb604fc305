// Host-side helpers shared by the C ABI's translation units: argument
// validation, the layer tag and the per-thread error message.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include "gdn.h"

namespace gdn_host {

// Records a printf-style message for gdn_last_error() on this host thread and returns st.
gdn_status fail(gdn_status st, const char *fmt, ...);
gdn_status cuda_fail(cudaError_t e, const char *what);
bool aligned16(const void *p);
int64_t channels(const gdn_layer_desc *d);          // conv channels: 2 Hk d_k + Hv d_v
size_t in_elt(const gdn_layer_desc *d);              // bytes per input element
gdn_status check_desc(const gdn_layer_desc *d);
uint64_t tag_of(const gdn_layer_desc *d);            // FNV-1a over the description (never 0)
gdn_status check_state(const gdn_layer_desc *d, const gdn_session *s, const char *what, bool need_present);

}  // namespace gdn_host
