// NVTX ranges in the "cc_dp" domain: one per C-ABI call, per bucket launch,
// and per arm and proxy-backward layer of the overlap measurement, so that a
// profiler timeline (or ncu --nvtx-include "cc_dp@...") can place the
// bucket launches against the compute stream -- the diagnosis the pages
// recommend for exposed communication ("Overlapping Communication and
// Computation": a profiler timeline of collective kernels against gaps in
// the compute stream).
//
// NVTX3 is header-only: with no profiler attached a range costs a call
// through a function pointer that returns at once; nothing is allocated
// and nothing is linked.  Ranges mark host enqueue time, not kernel time.
#pragma once

#include <cstdint>

#include <nvtx3/nvToolsExt.h>

namespace ccdp {

inline nvtxDomainHandle_t trace_domain() {
    static const nvtxDomainHandle_t domain = nvtxDomainCreateA("cc_dp");
    return domain;
}

// A range from construction to destruction; `payload` is a number shown
// with it (a bucket's first element, a layer index, an element count).
class TraceRange {
  public:
    explicit TraceRange(const char *name, uint64_t payload = 0) {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        a.payloadType = NVTX_PAYLOAD_TYPE_UNSIGNED_INT64;
        a.payload.ullValue = payload;
        nvtxDomainRangePushEx(trace_domain(), &a);
    }
    ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace ccdp
