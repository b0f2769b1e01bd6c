"""FP8-pool decode (sda_decode_fp8) on the GPU.

Element d of pool row s is e4m3(kv_fp8[s, d]) * kv_scale[s]; the reference is
the fp64 oracle of that pool (oracle.sda_decode_fp8).  With power-of-two row
scales (the workloads' quantisation) every dequantised element is exact in
bf16 and the bf16 path's tolerance applies unchanged.  Any other scale adds
one bf16 rounding of code * scale per element; that case is pinned instead
against the bf16 entry point on torch's bf16 dequantisation of the same pool,
which must give bit-identical outputs because both kernels then multiply the
same bf16 tile.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
import sink_sda_decode_gb300 as sda
from sink_sda_decode_gb300 import inputs

pytestmark = pytest.mark.gpu


def run_fp8(w, pool, sink=None, scale=None, workspace=None):
    idx, ptr = parity.to_dev(w)
    return sda.decode_fp8(w.q, pool.codes, pool.scale, idx, ptr,
                          w.attn_sink if sink is None else sink,
                          w.softmax_scale if scale is None else scale, workspace=workspace)


def oracle_fp8(w, pool, tokens=None, sink=None):
    codes, sc, idx, ptr = inputs.fp8_rows_for(w, pool, tokens)
    q = w.q_bits()
    if tokens is not None:
        q = q[np.asarray(tokens)]
    s = (w.attn_sink if sink is None else sink).cpu().numpy()
    return oracle.sda_decode_fp8(q, codes, sc, idx, ptr, s, w.softmax_scale)


def dequantised_bf16(pool):
    """bf16(code * scale) with torch (round to nearest even)."""
    return (pool.codes.view(torch.float8_e4m3fn).float() * pool.scale[:, None]).to(torch.bfloat16)


@pytest.mark.parametrize("cfg", range(1, len(inputs.CONFIG_NAMES)),
                         ids=inputs.CONFIG_NAMES[1:])
def test_workload_parity_fp8(cfg):
    """Every token of every workload against the FP8-pool oracle."""
    w = inputs.config(cfg, device="cuda")
    pool = inputs.fp8_pool(w)
    out = run_fp8(w, pool)
    torch.cuda.synchronize()
    ref = oracle_fp8(w, pool)
    st = parity.compare(out, ref)
    print(f"\n{inputs.CONFIG_NAMES[cfg]} fp8: {st}")
    parity.assert_parity(st, f"{inputs.CONFIG_NAMES[cfg]} fp8")
    zero = np.nonzero(w.lengths == 0)[0]
    if zero.size:
        assert torch.all(out[torch.from_numpy(zero).to(out.device)].view(torch.int16) == 0)


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_fp8_matches_bf16_path_on_the_dequantised_pool(H):
    """Same tile in shared memory -> the same output bits as sda_decode."""
    w = inputs.random_small(seed=60 + H, N=5, H=H, D=512, P=20000,
                            lengths=[0, 1, 63, 64, 700], device="cuda")
    pool = inputs.fp8_pool(w, pow2=False)  # scales max|row| / 448: products round in bf16
    a = run_fp8(w, pool)
    idx, ptr = parity.to_dev(w)
    b = sda.decode(w.q, dequantised_bf16(pool), idx, ptr, w.attn_sink, w.softmax_scale)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fp8_scales_zero_and_negative():
    """Rows with scale 0 (all-zero key and value) and negated rows (negative
    scale), over split long lists and two head groups; values stay unit
    normal, so the bf16 path's tolerance applies."""
    w = inputs.random_small(seed=71, N=4, H=128, D=512, P=1 << 16, lengths=[9000, 2, 0, 3000],
                            sink_sigma=1.5, device="cuda")
    pool = inputs.fp8_pool(w)
    g = torch.Generator(device="cuda").manual_seed(5)
    u = torch.rand(pool.scale.shape, generator=g, device="cuda")
    mult = torch.where(u < 0.1, 0.0, torch.where(u < 0.4, -1.0, 1.0))
    pool = inputs.Fp8Pool(codes=pool.codes, scale=pool.scale * mult)
    sink = w.attn_sink.clone()
    sink[3], sink[100] = -math.inf, math.inf
    out = run_fp8(w, pool, sink=sink)
    ref = oracle_fp8(w, pool, sink=sink)
    parity.assert_parity(parity.compare(out, ref), "fp8 scales")


def test_fp8_tail_tiles_and_duplicates():
    w = inputs.random_small(seed=72, N=6, H=64, D=512, P=300,
                            lengths=[1, 7, 65, 129, 250, 640], device="cuda", duplicates=True)
    pool = inputs.fp8_pool(w)
    parity.assert_parity(parity.compare(run_fp8(w, pool), oracle_fp8(w, pool)), "fp8 tails")


def test_fp8_rejects_unsupported_shapes_and_dtypes():
    w = inputs.random_small(seed=73, N=2, H=8, D=64, P=100, lengths=[3, 4], device="cuda")
    pool = inputs.fp8_pool(w)
    with pytest.raises(RuntimeError):
        run_fp8(w, pool)  # D = 64 has no FP8 path
    w = inputs.random_small(seed=74, N=2, H=16, D=512, P=100, lengths=[3, 4], device="cuda")
    pool = inputs.fp8_pool(w)
    idx, ptr = parity.to_dev(w)
    with pytest.raises(TypeError):
        sda.decode_fp8(w.q, pool.codes.to(torch.int32), pool.scale, idx, ptr, w.attn_sink, 1.0)
    with pytest.raises(ValueError):
        sda.decode_fp8(w.q, pool.codes, pool.scale[:-1], idx, ptr, w.attn_sink, 1.0)
    # float8 tensors are accepted as they are
    out = sda.decode_fp8(w.q, pool.codes.view(torch.float8_e4m3fn), pool.scale, idx, ptr,
                         w.attn_sink, w.softmax_scale)
    parity.assert_parity(parity.compare(out, oracle_fp8(w, pool)), "fp8 dtype")


def test_fp8_graph_capture_replay():
    w = inputs.random_small(seed=75, N=8, H=32, D=512, P=5000, lengths=[100] * 8, device="cuda")
    pool = inputs.fp8_pool(w)
    idx, ptr = parity.to_dev(w)
    ws = torch.empty(sda.workspace_size_fp8(w.N, w.H, w.D, idx.numel()), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sda.decode_fp8(w.q, pool.codes, pool.scale, idx, ptr, w.attn_sink, w.softmax_scale,
                       out=out, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sda.decode_fp8(w.q, pool.codes, pool.scale, idx, ptr, w.attn_sink, w.softmax_scale,
                       out=out, workspace=ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    parity.assert_parity(parity.compare(out, oracle_fp8(w, pool)), "fp8 graph")
