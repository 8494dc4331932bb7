"""The decode attention entry point that allocates nothing (collected last on purpose).

llama_attention_decode_static serves callers that cannot allocate device memory: its split
partials live in a fixed array inside the library instead of a caller workspace.  Two calls in
a row, on different inputs, must each agree with llama_attention_decode (the workspace form) on
the same inputs, within the bf16 tolerance of the other tests, and the fp64 oracle's attention on
those inputs (the cache slots each sequence sees, 0 .. positions[b]); an oversized request is
refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_dev):
    from llama_decoder_block_gb300 import build, api as a
    build.build()
    assert a.device_status() == 0
    return a


def _static(api, dims, q, kc, vc, pos, out):
    from llama_decoder_block_gb300 import _native as N
    d = dims.c()
    return N.lib().llama_attention_decode_static(ctypes.byref(d), q.data_ptr(), api.cache_struct(kc, vc),
                                                 pos.data_ptr(), out.data_ptr(), q.shape[0],
                                                 torch.cuda.current_stream().cuda_stream)


def test_fixed_scratch_decode_attention_matches_the_workspace_form(api):
    H, G, B, T_max = 32, 8, 16, 2100
    dims = api.Dims(H * 128, H, G, 128, 128, 1e-5, torch.bfloat16)
    ws = api.workspace(api.attention_decode_workspace_bytes(dims, B, T_max), "cuda")
    rng = np.random.default_rng(2024)
    for call in range(2):
        q = torch.from_numpy(rng.standard_normal((B, H, 128), dtype=np.float32)).cuda().to(torch.bfloat16)
        kc = torch.from_numpy(rng.standard_normal((B, G, T_max, 128), dtype=np.float32)).cuda().to(torch.bfloat16)
        vc = torch.from_numpy(rng.standard_normal((B, G, T_max, 128), dtype=np.float32)).cuda().to(torch.bfloat16)
        pos = torch.from_numpy(rng.integers(0, T_max, size=B).astype(np.int32)).cuda()
        pos[0] = 0
        pos[1] = T_max - 1
        ref = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
        api.attention_decode(dims, q, kc, vc, pos, ref, ws)
        got = torch.full_like(ref, float("nan"))
        assert _static(api, dims, q, kc, vc, pos, got) == 0
        assert api.device_status() == 0
        assert_close(f64(got), f64(ref), TOL["bf16"], f"fixed-scratch decode attention, call {call + 1}")
        # the oracle on the same bf16 inputs: one query per sequence at position pos[b], keys 0 .. pos[b]
        p64 = pos.cpu().numpy().astype(np.int64)
        want = oracle.attention(f64(q)[:, :, None, :], f64(kc), f64(vc), p64[:, None], p64 + 1)
        assert_close(f64(got), want[:, :, 0, :].reshape(B, H * 128), TOL["bf16"],
                     f"fixed-scratch decode attention vs oracle, call {call + 1}")


def test_fixed_scratch_refuses_requests_beyond_its_size(api):
    # (1024 * 8 + 256) segment slots * 4 heads * 130 floats > 16 MiB; the cache is real (small
    # T_max) so that the arguments are valid apart from the scratch size
    H, G, B, T_max = 32, 8, 1024, 16
    dims = api.Dims(H * 128, H, G, 128, 128, 1e-5, torch.bfloat16)
    q = torch.zeros(B, H, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(B, G, T_max, 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
    from llama_decoder_block_gb300 import _native as N
    d = dims.c()
    rc = N.lib().llama_attention_decode_static(ctypes.byref(d), q.data_ptr(), N.KVCache(kv.data_ptr(), kv.data_ptr(),
                                               T_max), pos.data_ptr(), out.data_ptr(), B, None)
    assert rc == -6
