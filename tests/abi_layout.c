/* Prints the sizes and field offsets of the C ABI structs, so that the
 * Python binding's ctypes mirrors can be checked against the header. */
#include <stddef.h>
#include <stdio.h>
#include "qg.h"

#define F(T, f) printf("%s.%s %zu\n", #T, #f, offsetof(T, f))
int main(void) {
    printf("qg_config %zu\n", sizeof(qg_config));
    F(qg_config, n_rot); F(qg_config, eps); F(qg_config, rope_theta); F(qg_config, layer_kinds);
    printf("qg_qtensor %zu\n", sizeof(qg_qtensor));
    F(qg_qtensor, qtype); F(qg_qtensor, n); F(qg_qtensor, k);
    printf("qg_layer_weights %zu\n", sizeof(qg_layer_weights));
    F(qg_layer_weights, ffn_gate); F(qg_layer_weights, ffn_down); F(qg_layer_weights, ssm_conv1d);
    F(qg_layer_weights, attn_qkv); F(qg_layer_weights, ssm_out); F(qg_layer_weights, attn_q_norm);
    F(qg_layer_weights, attn_q); F(qg_layer_weights, attn_output);
    printf("qg_host_weights %zu\n", sizeof(qg_host_weights));
    F(qg_host_weights, lm_head); F(qg_host_weights, layers);
    printf("qg_stats %zu\n", sizeof(qg_stats));
    F(qg_stats, graph_kernel_nodes); F(qg_stats, steps);
    return 0;
}
