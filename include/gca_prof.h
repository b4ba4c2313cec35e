/*
 * gca_prof.h -- optional per-kernel timing of the GCA library.
 *
 * When enabled on a host thread, every kernel the library launches from that
 * thread is bracketed by two CUDA events recorded on the launch stream, so
 * the device time of each kernel is measured on the stream it runs on.  Off
 * by default; costs two event records per launch when on.
 */
#ifndef GCA_PROF_H_
#define GCA_PROF_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Turn event bracketing on (1) or off (0) for the calling host thread. */
void gca_prof_enable(int on);

/*
 * Wait for the recorded events, then report per kernel name (at most `max`
 * names): names[i*64 .. i*64+63] (NUL-terminated), total_ms[i] (sum of the
 * event-to-event times) and launches[i].  Clears the records.  Returns the
 * number of names written, or -1 if a CUDA call failed.
 */
int gca_prof_read(int max, char* names, float* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* GCA_PROF_H_ */
