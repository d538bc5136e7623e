"""Host logic of CodecPath on the CPU (no kernel runs): the specs' sizes, the
buffers a pass allocates against the oracle's size rules, the checks on
inconsistent modes, the hpZ secondary-partition views, and the rotation of the
device input sets that the host-buffer pass takes turns over."""
import pytest
import torch

import oracle
from gradient_comm_codecs_gb300 import AdamSpec, CodecPath, QgzSpec, QwzSpec


def test_specs():
    q = QwzSpec(nranks=1, shard=1 << 28, block=2048, bits=8, chunks=27,
                tail_shard=7 * 10 ** 9 - 26 * (1 << 28))
    assert q.call_shards()[:-1] == [1 << 28] * 26
    assert q.phi == 7 * 10 ** 9
    g = QgzSpec(8, 8, 1 << 26, 256, 4)
    assert (g.nd, g.L) == (64, 1 << 20)
    assert AdamSpec(step=3).hparams() == (1e-4, 0.9, 0.999, 1e-8, 3)


def test_buffers_follow_the_size_rules():
    q = QwzSpec(nranks=4, shard=3 * 256 + 64, block=256, bits=8, nodes=2)
    g = QgzSpec(2, 2, 4 * 3 * 256, 256, 4)
    p = CodecPath(q, g, AdamSpec(), device="cpu", keep_grad=True, microbatches=2,
                  standalone_adam=1000, hpz=True)
    nd, b, L = g.nd, g.bucket, g.L
    assert p.w.numel() == p.w_full.numel() == q.phi and p.w.dtype == torch.bfloat16
    assert p.w_codes[0].numel() == q.nranks * oracle.codes_bytes(q.shard, 8)
    assert p.w_scales[0].numel() == q.nranks * oracle.num_blocks(q.shard, q.block)
    assert len(p.grads_mb) == 2 and p.grads is p.grads_mb[-1]
    assert p.acc.numel() == nd * b and p.acc.dtype == torch.float32
    assert p.msg1.numel() == nd * oracle.codes_bytes(b, 4)
    assert p.msg1_scales.numel() == nd * b // g.block
    assert p.msg2.numel() == nd * oracle.codes_bytes(g.nodes * L, 4)
    assert p.msg2_scales.numel() == nd * g.nodes * L // g.block
    assert p.grad_out.numel() == p.master.numel() == p.param.numel() == b
    assert p.sa_grad.numel() == p.sa_param.numel() == 1000
    # qwZ quant + dequant, the hpZ gather, one accumulation, reorder+quant, hop 1,
    # hop 2 with Adam, the standalone Adam
    assert p.launches_per_run == 2 + 1 + 1 + 2 + 1 + 1


def test_inconsistent_modes_are_rejected():
    q = QwzSpec(nranks=4, shard=768, block=256, bits=8)
    g = QgzSpec(2, 2, 4 * 768, 256, 4)
    with pytest.raises(ValueError):
        CodecPath(q, g, AdamSpec(), device="cpu", microbatches=0)
    with pytest.raises(ValueError):  # qwZ shards differ from the owned slices' block
        CodecPath(QwzSpec(4, 768, 512, 8), g, AdamSpec(), device="cpu", fuse_qwz=True)
    with pytest.raises(ValueError):
        CodecPath(q, g, None, device="cpu", fuse_qwz=True)
    with pytest.raises(ValueError):
        CodecPath(None, g, AdamSpec(), device="cpu", ring=True, microbatches=2)
    with pytest.raises(ValueError):
        CodecPath(QwzSpec(4, 768, 256, 8, chunks=2), g, AdamSpec(), device="cpu", hpz=True)
    with pytest.raises(ValueError):
        CodecPath(QwzSpec(4, 768, 256, 8, nodes=3), g, AdamSpec(), device="cpu", hpz=True)
    with pytest.raises(ValueError):
        CodecPath(q, g, None, device="cpu", standalone_adam=10)
    CodecPath(q, g, AdamSpec(), device="cpu", fuse_qwz=True)  # shards == owned slices


@pytest.mark.parametrize("N,G,bits", [(2, 4, 8), (4, 2, 4), (1, 8, 8)])
def test_secondary_partitions_tile_the_gathered_message(N, G, bits):
    shard, block = 2 * 512 + 128, 512
    p = CodecPath(QwzSpec(nranks=N * G, shard=shard, block=block, bits=bits, nodes=N), None,
                  None, device="cpu", hpz=True)
    codes, scales = p.secondary_partitions()
    assert len(codes) == len(scales) == G
    for c, s in zip(codes, scales):
        assert c.numel() + 4 * s.numel() == oracle.hpz_secondary_bytes(N, shard, block, bits)
    assert sum(c.numel() for c in codes) == p.w_codes[0].numel()
    assert codes[0].data_ptr() == p.w_codes[0].data_ptr()
    assert codes[-1].data_ptr() + codes[-1].numel() == p.w_codes[0].data_ptr() + p.w_codes[0].numel()


def test_input_set_rotation():
    q = QwzSpec(nranks=4, shard=768, block=256, bits=8)
    g = QgzSpec(2, 2, 4 * 768, 256, 4)
    p = CodecPath(q, g, AdamSpec(), device="cpu", microbatches=2, standalone_adam=100)
    w0, gm0, sa0 = p.w, p.grads_mb, p.sa_grad
    p._bind_input_set(0, 3, ())
    assert p.w is w0 and p.grads_mb is gm0 and p.sa_grad is sa0
    # set 1 for the inputs copied in; the others stay where they were
    p._bind_input_set(1, 3, ["w", "grads_mb"])
    assert p.w is not w0 and p.w.shape == w0.shape and p.w.dtype == w0.dtype
    assert p.grads_mb is not gm0 and len(p.grads_mb) == 2 and p.grads is p.grads_mb[-1]
    assert all(t.data_ptr() != u.data_ptr() for t, u in zip(p.grads_mb, gm0))
    assert p.sa_grad is sa0
    assert p._bound == {"w": 1, "grads_mb": 1, "sa_grad": 0}
    w1 = p.w
    p._bind_input_set(2, 3, ["w", "grads_mb", "sa_grad"])
    assert len({id(w0), id(w1), id(p.w)}) == 3 and p.sa_grad is not sa0
    p._bind_input_set(1, 3, ["w"])
    assert p.w is w1 and p._bound["w"] == 1
    # a new set count keeps set 0, the path's own buffers
    p._bind_input_set(0, 2, ["w", "grads_mb", "sa_grad"])
    assert p.w is w0 and p.grads_mb is gm0 and p.sa_grad is sa0 and len(p._sets) == 2
