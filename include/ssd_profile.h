/*
 * ssd_profile.h -- optional timing hook of the SSD library (measurement only; the
 * operation itself has no counterpart on the pages).
 *
 * While enabled (per host thread), every ssd_forward records a pair of CUDA events on
 * its stream around its dominant kernel (the one that reads x and writes y). The
 * events come from a pool the library creates on first use and keeps until exit;
 * no device memory is allocated. ssd_profile_read synchronises on the recorded events,
 * returns the summed elapsed time and the number of recorded launches, and resets
 * the pool for reuse. The library also counts every kernel it launches while recording.
 */
#ifndef SSD_GB300_PROFILE_H
#define SSD_GB300_PROFILE_H

#ifdef __cplusplus
extern "C" {
#endif

/* on != 0 enables recording for the calling host thread (starting a fresh record when it was
 * off); 0 stops recording and keeps the record for ssd_profile_read. Returns SSD_OK. */
int ssd_profile_enable(int on);

/* Sum of elapsed milliseconds over the recorded launches and their count; resets the
 * record. Returns SSD_OK, or SSD_ERR_CUDA if an event query fails. */
int ssd_profile_read(double *total_ms, int *launches);

/* Kernels of this library launched from the calling host thread since recording was last
 * enabled (all of them, not only the timed one). */
long long ssd_profile_kernel_launches(void);

/* Name of the kernel the events bracket (static string; "" before the first recorded call). */
const char *ssd_profile_kernel_name(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_GB300_PROFILE_H */
