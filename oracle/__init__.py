"""CPU oracle for the MoE expert-layer backward -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the GPU library computes, in float64 numpy,
written from the problem statements of three pages:

  * "Blockwise MM Backward MXFP8 Kernel API Reference" (parameters token_position_to_id,
    block_to_expert, block_size, gate_up_proj_act_checkpoint_T, the returned gradients and the
    "Dimensions" list with the block-count formula N),
  * "Matmul MXFP8 Backward Kernel API Reference" ("Forward pass convention": dX = dY @ W,
    dW = dY^T @ X; float8_dtype),
  * sonic-moe functional/backward.py (`_down_projection_backward_act` with its dSwiGLU epilogue
    `gemm_dgated`, `db2_and_ds_kernel`, `db1_kernel`, `_up_projection_backward_act/_weight`,
    `_down_projection_backward_weight`, `_token_broadcast_backward`).

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg may import it.  It shares
no code with the CUDA path under moe_expert_layer_routing_gb300/ and never imports it.

Modules:
  route_meta  -- expert histogram, offsets, stable grouped order, block padding, block-count bound
  mxfp8       -- FP8 e4m3/e5m2 codecs and OCP-MX E8M0 group quantisation (bit-exact)
  moe         -- MoE forward (for pins), BF16-path backward, MXFP8-path backward, sampled outputs
  linear      -- dense linear backward, BF16 and MXFP8

Parity pins (tests/test_oracle_*.py): finite differences, float64 torch autograd, the E=1/K=1/s=1
dense-MLP reduction, token-permutation invariance, closed-form inner-product identities, brute
force over tiny routings, torch's own float8 casts.  No function here is "parity unpinned".
"""
