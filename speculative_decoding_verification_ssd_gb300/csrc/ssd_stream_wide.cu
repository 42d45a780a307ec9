// ssd_stream_wide.cu -- the wide forms of the persistent streaming kernel
// (ssd_stream.cu), in which both consumer groups of a CTA work on each unit,
// compiled in their own translation unit so that the one-group forms build in
// parallel and carry none of their code.
#define SSD_STREAM_WIDE_TU 1
#include "ssd_stream.cu"
