/* A plain C client of libfa_splitkv: it includes only the public header,
 * links the shared library and checks the host-only entry points (version,
 * status strings, planner, workspace sizes, synchronous argument errors, the
 * kernel report), none of which touches a device. */
#include <stdio.h>
#include <string.h>

#include "fa_splitkv.h"

#define CHECK(c)                                                    \
  do {                                                              \
    if (!(c)) {                                                     \
      printf("FAIL %s:%d: %s\n", __FILE__, __LINE__, #c);           \
      return 1;                                                     \
    }                                                               \
  } while (0)

int main(void) {
  int ns = -1, units = -1;
  const void* dev = (const void*)0x10000; /* never dereferenced: the call fails first */
  const int* cu = (const int*)0x20000;

  CHECK(fa_version() > 0);
  CHECK(fa_status_string(FA_OK) != NULL && fa_status_string(FA_OK)[0] != '\0');
  CHECK(strcmp(fa_status_string(FA_ERR_INVALID_ARG), fa_status_string(FA_ERR_WORKSPACE)) != 0);

  /* planner: one query, 32 KV heads -> 32 units; the first split count whose
   * wave efficiency reaches 0.9 is 9 on 148 SMs (288/296) and on 152 (288/304) */
  CHECK(fa_plan(1, 1, 32, 32, 0, 148, &ns, &units) == FA_OK && ns == 9 && units == 32);
  CHECK(fa_plan(1, 1, 32, 32, 0, 152, &ns, &units) == FA_OK && ns == 9);
  /* enough units for two waves: one split; explicit counts clip at 128 */
  CHECK(fa_plan(8, 4096, 16, 16, 0, 152, &ns, &units) == FA_OK && ns == 1 && units == 4096);
  CHECK(fa_plan(1, 1, 32, 32, 500, 152, &ns, &units) == FA_OK && ns == 128);

  /* workspace: partials for several splits, the 16-byte tile counter for one */
  CHECK(fa_fwd_splitkv_workspace_size(3, 70, 12, 4, 128, 4) == (size_t)4 * 3 * 70 * 12 * 129 * 4);
  CHECK(fa_fwd_splitkv_workspace_size(1, 1, 32, 32, 128, 1) == 16);
  CHECK(fa_fwd_splitkv_workspace_size(1, 1, 3, 2, 128, 4) == 0); /* h_q % h_kv */

  /* argument errors are reported before anything is enqueued */
  CHECK(fa_fwd_splitkv_ex(dev, dev, dev, cu, cu, 1, 1, 1, 1, 6, 4, 128, 128, 0.f, 0, -1, 0,
                          (void*)dev, NULL, NULL, 0, FA_BF16, FA_BF16, NULL, NULL, NULL,
                          FA_KERNEL_AUTO, NULL) == FA_ERR_INVALID_ARG);
  CHECK(fa_fwd_splitkv_ex(dev, dev, dev, cu, cu, 1, 1, 1, 1, 4, 4, 96, 96, 0.f, 0, -1, 0,
                          (void*)dev, NULL, NULL, 0, FA_BF16, FA_BF16, NULL, NULL, NULL,
                          FA_KERNEL_AUTO, NULL) == FA_ERR_UNSUPPORTED);
  CHECK(fa_debug_last_kernel() == FA_KID_NONE);
  /* host-buffer call: its device-buffer size, and a missing buffer refused before any copy */
  CHECK(fa_fwd_splitkv_host_buffer_size(1, 1, 64, 1, 4, 4, 128, 128, FA_BF16, FA_BF16, 2) > 0);
  CHECK(fa_fwd_splitkv_host_buffer_size(1, 1, 64, 1, 6, 4, 128, 128, FA_BF16, FA_BF16, 2) == 0);
  CHECK(fa_fwd_splitkv_host(dev, dev, dev, cu, cu, 1, 1, 64, 1, 4, 4, 128, 128, 0.f, 0, -1, 2,
                            (void*)dev, NULL, NULL, 0, FA_BF16, FA_BF16, NULL, NULL, NULL, 0,
                            NULL) == FA_ERR_INVALID_ARG);

  puts("c client ok");
  return 0;
}
