"""plsh_alibi_attn_host: host-memory tensors give the device result bit for bit.

The host entry point stages Q, K, V through device buffers in query-row
chunks and copies O back while the kernel works on the next chunk; every
query tile is computed by the same kernel as on the device path, so the
results must be identical, whatever the chunking, the mask or the memory
kind.
"""
import pytest
import torch

import positional_lsh_approximation_gb300 as plsh
from positional_lsh_approximation_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, Hq, Hkv, n, d, dtype, causal, s, sigma, pinned
    ("causal_chunked", 2, 4, 2, 1000, 128, "bf16", True, 10, (1.2, 6.0, 40.0, 300.0), True),
    ("noncausal_chunked", 1, 2, 1, 777, 128, "bf16", False, 6, (3.0, 150.0), True),
    ("pageable", 1, 2, 1, 600, 128, "bf16", True, 7, (2.5, 90.0), False),
    ("single_tile", 1, 2, 1, 100, 128, "bf16", True, 4, (2.0, 20.0), True),
    ("simt_f32", 1, 2, 1, 300, 64, "f32", True, 5, (4.0, 30.0), True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_buffers_match_device(case):
    plsh.build()
    name, B, Hq, Hkv, n, d, dtype, causal, s, sig, pinned = case
    w = Workload(name, B, Hq, Hkv, n, d, dtype, causal, s, sig, qkv_seed=n + 11)
    Q, K, V = make_qkv(w)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    host = [torch.from_numpy(x).to(tdt) for x in (Q, K, V)]
    if pinned:
        host = [x.pin_memory() for x in host]
    dev = [x.cuda() for x in host]
    bins = plsh.sample_bins(n, w.sigmas(), s, seed=4)
    ref = plsh.alibi_attn(*dev, bins, causal)
    out = torch.full(host[0].shape, float("nan"), dtype=tdt)
    if pinned:
        out = out.pin_memory()
    got = plsh.alibi_attn_host(*host, bins, causal, out=out)
    torch.cuda.current_stream().synchronize()
    plsh.stream_status()
    assert got is out
    assert torch.equal(out, ref.cpu())
    # a second call reuses the staging buffers
    got2 = plsh.alibi_attn(*host, bins, causal)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(got2, ref.cpu())
    bins.free()
