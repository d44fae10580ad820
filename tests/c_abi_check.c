/* A plain C99 caller of the library: the header compiles as C, the shared library
 * links, and the calls that need no GPU behave as the header states (sizes, argument
 * rejection, status names, the staging copy).  Prints "ok" and exits 0 on success. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dllm_cache.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      fprintf(stderr, "check failed line %d: %s\n", __LINE__, #c); \
      return 1;                                               \
    }                                                         \
  } while (0)

int main(void) {
  dllm_cache_desc d;
  memset(&d, 0, sizeof d);
  d.n_layers = 2;
  d.batch = 4;
  d.max_pos = 256;
  d.tail_slots = 16;
  d.n_heads = 8;
  d.head_dim = 128;
  d.kv_dtype = DLLM_E4M3;
  d.rope_theta = 500000.0;
  /* e4m3: one byte per element plus one fp32 scale per (slot, K|V, head) */
  const size_t slots = 256 + 16;
  CHECK(dllm_cache_bytes(&d) == 2u * 4u * slots * (2u * 8u * 128u + 2u * 8u * 4u));
  d.head_dim = 64; /* the tensor-core paths need 128 */
  CHECK(dllm_cache_bytes(&d) == 0);
  dllm_cache* c = (dllm_cache*)1;
  CHECK(dllm_cache_alloc(&d, &c) == DLLM_EUNSUPPORTED && c == NULL);
  d.head_dim = 128;
  d.batch = 0;
  CHECK(dllm_cache_alloc(&d, &c) == DLLM_EINVAL && c == NULL);
  CHECK(dllm_cache_free(NULL) == DLLM_OK);
  CHECK(dllm_cache_step(NULL, 0, NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL, 0, NULL, NULL) == DLLM_EINVAL);

  CHECK(strcmp(dllm_strerror(DLLM_OK), "ok") == 0);
  CHECK(strlen(dllm_strerror(DLLM_EDEVICE)) > 0 && strlen(dllm_strerror(12345)) > 0);

  /* staging copy: a byte copy at odd alignments, overlap rejected */
  unsigned char src[301], dst[320];
  for (int i = 0; i < 301; ++i) src[i] = (unsigned char)(i * 7 + 3);
  memset(dst, 0xA5, sizeof dst);
  CHECK(dllm_host_stage(dst + 3, src + 1, 300) == DLLM_OK);
  CHECK(memcmp(dst + 3, src + 1, 300) == 0 && dst[2] == 0xA5 && dst[303] == 0xA5);
  CHECK(dllm_host_stage(dst, dst + 8, 16) == DLLM_EINVAL);
  CHECK(dllm_host_stage(NULL, src, 0) == DLLM_OK);
  void* p = (void*)1;
  CHECK(dllm_host_alloc(0, &p) == DLLM_OK && p == NULL);
  CHECK(dllm_host_free(NULL) == DLLM_OK);
  puts("ok");
  return 0;
}
