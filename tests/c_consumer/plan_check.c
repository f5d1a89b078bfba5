/* A plain C99 consumer of the library's C ABI: it includes the public header
 * only, builds a plan for the dense decode workload's shape on the host (no
 * GPU call), checks the result codes, the workspace layout and the error
 * strings, and calls the run / combine entry points with arguments they
 * reject before any CUDA call.  Exit status 0 on success. */
#include <stdio.h>
#include <string.h>

#include "mla_decode.h"

static int fail(const char* what) {
  fprintf(stderr, "plan_check: %s\n", what);
  return 1;
}

int main(void) {
  mla_problem pr;
  mla_plan plan;
  int32_t seq[4] = {100, 1000, 64, 0};
  size_t ws_bytes = 0;
  void* fake = (void*)(uintptr_t)(1u << 20);   /* aligned, never dereferenced */
  float* fake_f = (float*)fake;
  const int32_t* fake_i = (const int32_t*)fake;
  int rc;
  memset(&pr, 0, sizeof(pr));
  pr.batch = 4;
  pr.q_len = 1;
  pr.num_heads = 20;
  pr.kv_lora_rank = 512;
  pr.rope_dim = 64;
  pr.nope_dim = 192;
  pr.v_head_dim = 256;
  pr.page_size = 64;
  pr.num_pages = 100;
  pr.max_pages_per_seq = 30;
  pr.kv_dtype = MLA_KV_BF16;
  pr.topk_width = 0;
  pr.causal = 1;
  pr.sm_scale = 1.0f / 16.0f;
  rc = mla_decode_plan(&pr, seq, 152, 0, &plan, &ws_bytes);
  if (rc != MLA_OK) return fail(mla_strerror(rc));
  if (plan.num_streams != 4 || plan.planned_tiles != 2 + 16 + 1 + 0) return fail("row sets / tiles");
  if (plan.workspace_bytes <= plan.ws_status || plan.smem_bytes > 232448) return fail("layout");
  if (ws_bytes != (size_t)plan.workspace_bytes) return fail("workspace_bytes out-parameter");
  /* run and combine check the workspace size before anything is queued */
  if (mla_decode_run(&plan, fake, NULL, fake, fake_i, fake_i, NULL, fake, ws_bytes - 1, fake_f,
                     fake_f, NULL) != MLA_ERR_WORKSPACE_TOO_SMALL)
    return fail("short workspace accepted by mla_decode_run");
  if (mla_combine(&plan, fake_i, fake, 256, fake, fake_f, fake_f, fake, NULL) !=
      MLA_ERR_WORKSPACE_TOO_SMALL)
    return fail("short workspace accepted by mla_combine");
  if (mla_combine(&plan, fake_i, fake, ws_bytes, fake, fake_f, fake_f, NULL, NULL) !=
      MLA_ERR_INVALID_ARGUMENT)
    return fail("W_UV without an output accepted");
  /* split-KV by length: 19 tiles at 512 tokens (8 tiles) per CTA -> 3 CTAs */
  rc = mla_decode_plan(&pr, seq, 152, 512, &plan, NULL);
  if (rc != MLA_OK || plan.num_ctas != 3) return fail("split_tokens");
  pr.q_len = 2;   /* two drafts of 20 heads share a row set */
  rc = mla_decode_plan(&pr, seq, 152, 0, &plan, NULL);
  if (rc != MLA_OK || plan.num_streams != 4) return fail("grouped drafts");
  pr.page_size = 96;
  if (mla_decode_plan(&pr, seq, 152, 0, &plan, NULL) != MLA_ERR_UNSUPPORTED)
    return fail("page 96 accepted");
  if (mla_decode_plan(NULL, seq, 152, 0, &plan, NULL) != MLA_ERR_INVALID_ARGUMENT)
    return fail("null problem");
  if (strcmp(mla_strerror(MLA_ERR_MISALIGNED), "device pointer not 16-byte aligned") != 0)
    return fail("strerror");
  if (mla_version() <= 0) return fail("version");
  printf("plan_check ok (ABI version %d)\n", mla_version());
  return 0;
}
