"""GB300-native ZeRO++ data-parallel codec path.

qwZ block quantization of weight shards, qgZ slice reorder + one-shot
quantization + two-hop hierarchical reduce, and the sharded mixed-precision
Adam step, as hand-written sm_103a CUDA kernels behind the C ABI of
``include/zpp.h`` (``libzpp.so``).  The functions here are that ABI with the
same names; ``CodecPath`` holds the buffers of one simulated multi-rank step.
"""
from ._lib import (  # noqa: F401
    EXPORTS, ZPP_ERR_CUDA, ZPP_ERR_INVALID_ARG, ZPP_ERR_MISALIGNED, ZPP_ERR_UNSUPPORTED, ZPP_OK,
    ZppError, library_path, zpp_abi_version, zpp_adam_hparams, zpp_adam_state, zpp_codes_bytes,
    zpp_grad_accumulate, zpp_hpz_gather, zpp_hpz_secondary_bytes, zpp_num_blocks, zpp_qgz_final_hop_adam_qwz, zpp_qgz_hop_reduce,
    zpp_qgz_reorder_quant, zpp_qgz_reorder_quant_acc, zpp_qgz_slice_perm, zpp_qwz_dequant,
    zpp_qwz_quant, zpp_ring_rs_step, zpp_shard_adam_step, zpp_status_string,
)
from .path import AdamSpec, CodecPath, QgzSpec, QwzSpec  # noqa: F401
