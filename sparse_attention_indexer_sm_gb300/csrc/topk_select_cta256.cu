// The 256-thread build of the top-k kernels (namespace topk_gb300::cta256); see
// topk_select.cu.
#define TOPK_CTA_THREADS 256
#include "topk_select.cu"
