"""The C-ABI calls inside a captured CUDA graph: ln_fwd, ln_bwd (with its
workspace and the programmatically launched finalize), ln_fwd_from_partials
and ln_softmax_fwd are captured once, the graph is replayed on new inputs
copied into the same buffers, and every output must equal, bit for bit,
eager calls on those inputs (same kernels, same deterministic partial
order)."""

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


TILE = 128


def _with_partials(inp):
    """Per-128-column-tile (sum, M2) partials of x, from torch ops (input data
    for ln_fwd_from_partials, standing in for a producing GEMM's epilogue)."""
    x = inp["x"].float()
    R, H = x.shape
    T = -(-H // TILE)
    t = torch.nn.functional.pad(x, (0, T * TILE - H)).view(R, T, TILE)
    n = torch.full((T,), float(TILE), device=x.device)
    n[-1] = H - (T - 1) * TILE
    psum = t.sum(-1)
    mask = (torch.arange(T * TILE, device=x.device) < H).view(T, TILE).float()
    psq = (((t - (psum / n)[..., None]) * mask) ** 2).sum(-1)
    inp["psum"], inp["psq"] = psum.contiguous(), psq.contiguous()
    return inp


# The two bench shapes, and widths that take the other backward layouts: two
# 64- or 128-thread row groups per CTA (1536, 2560), one 384-thread group
# per CTA with every column sum in more than 48 KiB of shared memory (12288).
@pytest.mark.parametrize("base", [
    W.BENCH_LN_BF16_576000x384, W.BENCH_RMS_BF16_16384x8192,
    W.BENCH_RMS_BF16_16384x8192.with_(name="rms_bf16_x1536", hidden=1536),
    W.BENCH_LN_BF16_576000x384.with_(name="ln_bf16_x2560", hidden=2560),
    W.BENCH_LN_BF16_576000x384.with_(name="ln_bf16_x12288", hidden=12288),
    W.BENCH_LN_BF16_576000x384.with_(name="ln_bf16_x16384", hidden=16384),
], ids=lambda w: w.name)
def test_fwd_bwd_softmax_replay_in_a_cuda_graph(cuda_lib, base):
    nf = cuda_lib
    w = base.with_(rows=4099 if base.hidden <= 1024 else 257)
    dev = torch.device("cuda")
    dt = W.TORCH_DTYPES[w.dtype]
    R, H = w.rows, w.hidden
    rms = w.mode == W.RMSNORM

    def buffers():
        inp = {k: (v.to(dev) if v is not None else None) for k, v in W.make_inputs(w, seed=1).items()}
        inp = _with_partials(inp)
        f32 = dict(dtype=torch.float32, device=dev)
        out = dict(sum=torch.empty(R, H, dtype=dt, device=dev), y=torch.empty(R, H, dtype=dt, device=dev),
                   mean=None if rms else torch.empty(R, **f32), rstd=torch.empty(R, **f32),
                   amax=torch.empty(1, **f32), dx=torch.empty(R, H, dtype=dt, device=dev),
                   dgamma=torch.empty(H, **f32), dbeta=None if rms else torch.empty(H, **f32),
                   sm=torch.empty(R, H, dtype=dt, device=dev),
                   py=torch.empty(R, H, dtype=dt, device=dev),
                   pmean=None if rms else torch.empty(R, **f32), prstd=torch.empty(R, **f32))
        ws = torch.empty(max(16, nf.ln_bwd_workspace_bytes(R, H, dt, w.mode)), dtype=torch.uint8,
                         device=dev)
        return inp, out, ws

    def step(inp, out, ws, stream):
        nf.ln_fwd(inp["x"], inp["bias"], inp["residual"], inp["gamma"], inp["beta"], w.eps, w.mode,
                  w.zero_centered_gamma, out["sum"], out["y"], out["mean"], out["rstd"], out["amax"],
                  stream)
        nf.ln_bwd(inp["dy"], out["sum"], inp["gamma"], out["mean"], out["rstd"], out["dx"],
                  out["dgamma"], out["dbeta"], stream, mode=w.mode,
                  zero_centered_gamma=w.zero_centered_gamma, workspace=ws)
        nf.ln_softmax_fwd(out["y"], out["sm"], stream)
        nf.ln_fwd_from_partials(inp["x"], inp["psum"], inp["psq"], TILE, "sum_m2", inp["gamma"],
                                inp["beta"], w.eps, w.mode, w.zero_centered_gamma, out["py"],
                                out["pmean"], out["prstd"], None, stream)

    inp, out, ws = buffers()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(inp, out, ws, s)          # warm up (plans, attributes) outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(inp, out, ws, torch.cuda.current_stream())

    # new inputs into the captured buffers, replay
    fresh = _with_partials({k: (v.to(dev) if v is not None else None)
                            for k, v in W.make_inputs(w, seed=2).items()})
    for k, v in fresh.items():
        if v is not None:
            inp[k].copy_(v)
    g.replay()
    torch.cuda.synchronize()

    inp2, out2, ws2 = buffers()
    for k, v in fresh.items():
        if v is not None:
            inp2[k].copy_(v)
    step(inp2, out2, ws2, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert nf.ln_device_error() == 0
    for k in out:
        if out[k] is not None:
            assert torch.equal(_bits(out[k]), _bits(out2[k])), k
