"""The full-size workloads, in the launch configuration the benchmark times,
checked on sampled channels against the fp64 oracle (channels are
independent, so a sampled channel's oracle is exact), plus the size-
independent identities (host-split calls equal one call bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, oracle_scan, sample_channels, sample_scan_inputs
from selective_state_space_118_b300 import inputs, ops

pytestmark = pytest.mark.gpu


def run_gpu(inp, **kw):
    return ops.mamba_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"],
                              inp["A_log"], inp["Dskip"], inp["conv_w"], inp.get("conv_b"),
                              inp.get("h0"), inp.get("conv_state0"), **kw)


def check_sampled(inp, outs, cs, io, what):
    y, fh, fcs = outs
    idx = torch.as_tensor(cs, device=y.device)
    yr, fhr, fcsr = oracle_scan(sample_scan_inputs(inp, cs))
    assert_close(y.index_select(2, idx), yr, io, f"{what} y")
    assert_close(fh.index_select(1, idx), fhr, io, f"{what} final_h", fp32_output=True)
    np.testing.assert_array_equal(oracle.f64(fcs.index_select(2, idx)), fcsr)


def test_jamba_prefill_full_size():
    w = inputs.JAMBA_PREFILL
    inp = inputs.workload_inputs(w, device="cuda")
    outs = run_gpu(inp)  # default plan, as timed by the benchmark
    torch.cuda.synchronize()
    check_sampled(inp, outs, sample_channels(w.d_inner, 48), w.io, w.name)


def test_prefill_256k_host_chunks_equal_one_pass():
    w = inputs.PREFILL_256K
    inp = inputs.workload_inputs(w, device="cuda")
    step = w.seqlen // w.host_chunks

    def split_calls(n_chunks):
        ys = torch.empty_like(inp["x"])
        h, cs = None, None
        for i in range(w.host_chunks):
            part = dict(inp, h0=h, conv_state0=cs)
            for k in ("x", "z", "dt_raw", "Bm", "Cm"):
                part[k] = inp[k][:, i * step:(i + 1) * step]
            _, h, cs = run_gpu(part, y=ys[:, i * step:(i + 1) * step], n_chunks=n_chunks)
        return ys, h, cs

    # one sequential pass == the same sequence as 64 calls of 4096 tokens with
    # the state carried between them, bit for bit
    y, fh, fcs = run_gpu(inp, n_chunks=1)
    ys, h, cs = split_calls(1)
    torch.cuda.synchronize()
    assert torch.equal(ys, y)
    assert torch.equal(h, fh) and torch.equal(cs, fcs)
    del ys
    cs12 = sample_channels(w.d_inner, 12)
    check_sampled(inp, (y, fh, fcs), cs12, w.io, w.name)
    del y
    # the default (chunked) plan, in one call and in 64 carried calls
    outs = run_gpu(inp)
    torch.cuda.synchronize()
    check_sampled(inp, outs, cs12, w.io, w.name + " default plan")
    del outs
    outs = split_calls(0)
    torch.cuda.synchronize()
    check_sampled(inp, outs, cs12, w.io, w.name + " default plan, 64 carried calls")


def test_decode_28_layers_full_size():
    w = inputs.DECODE
    rng = np.random.default_rng(0)
    bs = np.sort(rng.choice(w.batch, 4, replace=False))
    cs = sample_channels(w.d_inner, 16)
    bi = torch.as_tensor(bs, device="cuda")
    ci = torch.as_tensor(cs, device="cuda")
    for layer in range(w.layers):
        st = inputs.decode_layer_state(w, layer, device="cuda")
        tok = inputs.decode_token_inputs(w, layer, w.steps, device="cuda")
        sub = lambda t: t.index_select(0, bi).index_select(-1, ci)  # noqa: E731
        h_ref = oracle.f64(st["h"].index_select(0, bi).index_select(1, ci))
        cs_ref = oracle.f64(sub(st["conv_state"]))
        prm = [st[k].index_select(0, ci) for k in ("A_log", "Dskip", "conv_w", "conv_b")]
        ys = []
        for t in range(w.steps):
            y = ops.mamba_step(st["h"], st["conv_state"], tok["x_t"][t], tok["z_t"][t],
                               tok["dt_raw_t"][t], tok["B_t"][t], tok["C_t"][t], st["A_log"],
                               st["Dskip"], st["conv_w"], st["conv_b"])
            ys.append(sub(y))
        ys = torch.stack(ys).cpu()
        torch.cuda.synchronize()
        if layer % 7 == 0 or layer == w.layers - 1:  # oracle on a spread of layers
            for t in range(w.steps):
                yr, h_ref, cs_ref = oracle.step(
                    h_ref, cs_ref, sub(tok["x_t"][t]), sub(tok["z_t"][t]), sub(tok["dt_raw_t"][t]),
                    tok["B_t"][t].index_select(0, bi), tok["C_t"][t].index_select(0, bi), *prm)
                assert_close(ys[t], yr, w.io, f"layer {layer} step {t} y")
            assert_close(st["h"].index_select(0, bi).index_select(1, ci), h_ref, w.io,
                         f"layer {layer} h", fp32_output=True)
            np.testing.assert_array_equal(oracle.f64(sub(st["conv_state"])), cs_ref)
        del st, tok
