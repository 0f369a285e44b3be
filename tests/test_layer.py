"""Stride-aware calls and one attention layer around them (research.dws.rip/llm/kernels,
section 06 and Fig. 8: an attention layer plus a small loss, forward and backward,
replayed as a CUDA graph).

- The attention on strided views (q, k, v as head ranges of one fused QKV
  buffer; out, dout, dq, dk, dv as views into wider buffers) gives bit for bit
  what it gives on dense copies.
- The layer (QKV projection, attention, output projection, loss = sum(y * g),
  and the whole backward) against a float64 CPU reference: torch CPU float64
  matmuls for the projections and the oracle for the attention, fed the GPU's
  own bf16 intermediates so that each stage is compared on equal inputs.
- The layer step captured once in a CUDA graph with cu_seqlens padded to 42
  segments, replayed on three batches with different boundaries, equals eager
  steps bit for bit.
"""
import numpy as np
import pytest

import oracle
from varlen_sliding_window_gb300 import synth

from helpers import TOL_GRAD, TOL_OUT, rel_l2, to_device_bf16

pytestmark = pytest.mark.gpu


def test_strided_views_match_dense_bitwise():
    import torch
    from varlen_sliding_window_gb300 import binding
    cu = np.array([0, 1, 130, 386, 387, 900, 1024, 1536, 1800], dtype=np.int32)
    T, hq, hkv = 1800, 8, 2
    inp = synth.make_inputs(cu, hq, hkv, 128, tensor_seed=7)
    q, k, v, do = (to_device_bf16(b) for b in (inp.q_bits, inp.k_bits, inp.v_bits, inp.dout_bits))
    dcu = torch.from_numpy(cu).cuda()
    for window in (-1, 300):
        # Dense reference.
        out = torch.empty_like(q)
        lse = torch.empty(hq, T, dtype=torch.float32, device="cuda")
        binding.attn_varlen_fwd(q, k, v, dcu, 600, window, 0.0884, out, lse)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        binding.attn_varlen_bwd(do, q, k, v, out, lse, dcu, 600, window, 0.0884, dq, dk, dv)
        # Views: q, k, v inside one [T, 12, 128] buffer; out, dout in [T, 8, 256]
        # rows; dq, dk, dv inside one [T, 12, 128] gradient buffer.
        qkv = torch.cat([q, k, v], dim=1)
        qs, ks, vs = qkv[:, :hq], qkv[:, hq:hq + hkv], qkv[:, hq + hkv:]
        wide_out = torch.full((T, hq, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        outs = wide_out[:, :, 128:]
        wide_do = torch.zeros((T, hq, 256), dtype=torch.bfloat16, device="cuda")
        wide_do[:, :, :128] = do
        dos = wide_do[:, :, :128]
        lse2 = torch.empty_like(lse)
        binding.attn_varlen_fwd(qs, ks, vs, dcu, 600, window, 0.0884, outs, lse2)
        dqkv = torch.full((T, hq + 2 * hkv, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        dqs, dks, dvs = dqkv[:, :hq], dqkv[:, hq:hq + hkv], dqkv[:, hq + hkv:]
        binding.attn_varlen_bwd(dos, qs, ks, vs, outs, lse2, dcu, 600, window, 0.0884, dqs, dks, dvs)
        torch.cuda.synchronize()
        assert binding.attn_varlen_get_status() == 0
        for a, b in ((out, outs), (lse, lse2), (dq, dqs), (dk, dks), (dv, dvs)):
            assert torch.equal(a, b)
        # The untouched halves of the wide output rows stay NaN.
        assert torch.isnan(wide_out[:, :, :128].float()).all()


def _layer(cu, seed, d_model=256, hq=8, hkv=2, window=-1, nseg=None, max_seqlen=None):
    import torch
    from varlen_sliding_window_gb300.layer import AttentionLayer
    T = int(cu[-1])
    nseg = nseg or len(cu) - 1
    lay = AttentionLayer(T, d_model, hq, hkv, max_seqlen=max_seqlen or int(np.diff(cu).max()), window_left=window,
                         num_segments=nseg, seed=seed)
    gen = torch.Generator(device="cpu").manual_seed(seed + 1)
    lay.x.copy_(torch.randn(T, d_model, generator=gen).to(torch.bfloat16))
    lay.g.copy_(torch.randn(T, d_model, generator=gen).to(torch.bfloat16))
    lay.cu.copy_(torch.from_numpy(synth.pad_cu_seqlens(cu, nseg)))
    return lay


@pytest.mark.parametrize("window", [-1, 64])
def test_layer_against_float64_reference(window):
    import torch
    from varlen_sliding_window_gb300 import binding
    cu = np.array([0, 61, 161, 256], dtype=np.int32)
    lay = _layer(cu, seed=3, window=window)
    lay.step()
    torch.cuda.synchronize()
    assert binding.attn_varlen_get_status() == 0
    f64 = lambda t: t.detach().double().cpu()  # noqa: E731
    x, g, wq, wo = f64(lay.x), f64(lay.g), f64(lay.w_qkv), f64(lay.w_o)
    T, hq, hkv = 256, 8, 2
    qkv = f64(lay.qkv)
    assert rel_l2(qkv.numpy(), (x @ wq).view(T, -1, 128).numpy()) <= 1e-2
    q, k, v = qkv[:, :hq].numpy(), qkv[:, hq:hq + hkv].numpy(), qkv[:, hq + hkv:].numpy()
    ref_out, _ = oracle.forward(q, k, v, cu, window, lay.scale)
    out = f64(lay.out)
    assert rel_l2(out.numpy(), ref_out) <= TOL_OUT
    y = out.view(T, -1) @ wo
    assert rel_l2(f64(lay.y).numpy(), y.numpy()) <= 1e-2
    assert abs(float(lay.loss) - float((f64(lay.y) * g).sum())) <= 1e-3 * float((f64(lay.y).abs() * g.abs()).sum())
    d_out = f64(lay.d_out)
    assert rel_l2(d_out.view(T, -1).numpy(), (g @ wo.t()).numpy()) <= 1e-2
    assert rel_l2(f64(lay.dw_o).numpy(), (out.view(T, -1).t() @ g).numpy()) <= 1e-2
    dq, dk, dv = oracle.backward(d_out.numpy(), q, k, v, cu, window, lay.scale)
    d_qkv = f64(lay.d_qkv)
    for got, ref in ((d_qkv[:, :hq], dq), (d_qkv[:, hq:hq + hkv], dk), (d_qkv[:, hq + hkv:], dv)):
        assert rel_l2(got.numpy(), ref) <= TOL_GRAD
    assert rel_l2(f64(lay.dw_qkv).numpy(), (x.t() @ d_qkv.view(T, -1)).numpy()) <= 1e-2
    assert rel_l2(f64(lay.dx).numpy(), (d_qkv.view(T, -1) @ wq.t()).numpy()) <= 1e-2


def test_layer_graph_replay_matches_eager():
    import torch
    from varlen_sliding_window_gb300 import binding
    batches = [synth.pack_microbatch(16384, 4096, s) for s in (0, 1, 2)]
    lay = _layer(batches[0], seed=5, d_model=1024, nseg=42, max_seqlen=4096)
    names = ("qkv", "out", "lse", "y", "loss", "d_out", "d_qkv", "dw_qkv", "dw_o", "dx")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lay.step()  # outside capture first (library set-up, cuBLAS handles)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lay.step()
    for cu in batches:
        lay.cu.copy_(torch.from_numpy(synth.pad_cu_seqlens(cu, 42)))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        replayed = {n: getattr(lay, n).clone() for n in names}
        lay.step()
        torch.cuda.synchronize()
        for n in names:
            assert torch.equal(replayed[n], getattr(lay, n)), n
    assert binding.attn_varlen_get_status() == 0
