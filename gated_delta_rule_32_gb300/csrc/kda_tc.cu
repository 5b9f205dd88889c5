// kda_tc.cu -- tensor-core (tcgen05/TMEM/TMA) fused KDA forward.
#include "kda_common.cuh"

bool kda_tc_supported(int dk, int dv) { (void)dk; (void)dv; return false; }

kda_status kda_launch_tc(const kda::FwdParams& p, cudaStream_t stream) {
  (void)p; (void)stream;
  return KDA_ERR_UNSUPPORTED;
}

extern "C" kda_status kda_debug_intra(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      const uint16_t* g_logit, const uint16_t* beta, int B,
                                      int T, int H, int dk, int dv, const int32_t* cu_seqlens,
                                      int n, int h, float* gam, float* aqk, float* akk,
                                      float* tinv, float* w, float* u, kda_stream_t stream) {
  (void)q; (void)k; (void)v; (void)g_logit; (void)beta; (void)B; (void)T; (void)H; (void)dk;
  (void)dv; (void)cu_seqlens; (void)n; (void)h; (void)gam; (void)aqk; (void)akk; (void)tinv;
  (void)w; (void)u; (void)stream;
  return KDA_ERR_UNSUPPORTED;
}
