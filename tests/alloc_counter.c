/*
 * Counts the device-memory allocation and release calls that reach the CUDA
 * driver in this process, through CUPTI's callback API.
 *
 * TEST INFRASTRUCTURE: the allocation-free entry point's test compiles this
 * file and loads it into a child process before any CUDA call, so that it
 * sees every allocation the library under test makes -- including those of a
 * statically linked CUDA runtime, whose calls all pass through the driver.
 *
 *   int  alloc_counter_start(void)   subscribe; 0 on success, else the
 *                                    CUptiResult of the failing call
 *   long alloc_counter_allocs(void)  driver allocation calls seen so far
 *   long alloc_counter_frees(void)   driver release calls seen so far
 */
#include <cupti.h>

static long g_allocs;
static long g_frees;
static CUpti_SubscriberHandle g_subscriber;

static void CUPTIAPI on_driver_call(void* userdata, CUpti_CallbackDomain domain, CUpti_CallbackId cbid,
                                    const void* cbdata)
{
    const CUpti_CallbackData* d = (const CUpti_CallbackData*)cbdata;
    (void)userdata;
    if (domain != CUPTI_CB_DOMAIN_DRIVER_API || d->callbackSite != CUPTI_API_ENTER) return;
    switch (cbid) {
    case CUPTI_DRIVER_TRACE_CBID_cuMemAlloc:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAlloc_v2:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocPitch:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocPitch_v2:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocManaged:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocAsync:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocAsync_ptsz:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocFromPoolAsync:
    case CUPTI_DRIVER_TRACE_CBID_cuMemAllocFromPoolAsync_ptsz:
    case CUPTI_DRIVER_TRACE_CBID_cuMemCreate:
        __atomic_add_fetch(&g_allocs, 1, __ATOMIC_SEQ_CST);
        break;
    case CUPTI_DRIVER_TRACE_CBID_cuMemFree:
    case CUPTI_DRIVER_TRACE_CBID_cuMemFree_v2:
    case CUPTI_DRIVER_TRACE_CBID_cuMemFreeAsync:
    case CUPTI_DRIVER_TRACE_CBID_cuMemRelease:
        __atomic_add_fetch(&g_frees, 1, __ATOMIC_SEQ_CST);
        break;
    default:
        break;
    }
}

int alloc_counter_start(void)
{
    CUptiResult r = cuptiSubscribe(&g_subscriber, (CUpti_CallbackFunc)on_driver_call, 0);
    if (r != CUPTI_SUCCESS) return (int)r;
    r = cuptiEnableDomain(1, g_subscriber, CUPTI_CB_DOMAIN_DRIVER_API);
    return (int)r;
}

long alloc_counter_allocs(void) { return __atomic_load_n(&g_allocs, __ATOMIC_SEQ_CST); }

long alloc_counter_frees(void) { return __atomic_load_n(&g_frees, __ATOMIC_SEQ_CST); }
