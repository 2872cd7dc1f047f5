// Optional per-CTA phase timestamps (%globaltimer) for studying where a
// kernel's time goes.  Compiled out unless SSD_TRACE is defined; a traced
// build links a device array g_ssd_trace[kernel][cta][event] (relocatable
// device code) that the caller reads back after a call.
#pragma once

#ifdef SSD_TRACE
extern __device__ unsigned long long g_ssd_trace[];
// Event 0 records %globaltimer (ns, comparable across CTAs) and, in slot 30,
// the SM cycle counter; later events record the SM cycle counter only, so
// phase lengths inside a CTA are exact.  Slot 31 holds the SM id.
__device__ __forceinline__ void ssd_trace_event(int kernel, int ev)
{
    const unsigned cta = blockIdx.x + blockIdx.y * gridDim.x;
    if (cta >= 8192u || ev >= 30)
        return;
    unsigned long long *rec = g_ssd_trace + (static_cast<unsigned long long>(kernel) * 8192u + cta) * 32u;
    const unsigned long long c = clock64();
    if (ev == 0) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        rec[0] = t;
        rec[30] = c;
        rec[31] = smid;
    } else {
        rec[ev] = c;
    }
}
#define SSD_TRACE_EV(k, e) ssd_trace_event((k), (e))
#else
#define SSD_TRACE_EV(k, e) ((void)0)
#endif
