"""The allocation-free sampler entry point against the regular one (GPU).

reset_sample_noalloc serves callers that cannot allocate device memory (an
engine that owns all device memory, a decode loop that must not call
cudaMalloc); it keeps its scratch in a static device array instead of a
caller workspace.  It must give the same tokens, entropies and temperatures as
reset_sample, call after call, since the array keeps the previous call's
contents.  Both are called through the C ABI.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_w4a4_decode_gemv_gb300 import synth
from nvfp4_w4a4_decode_gemv_gb300._lib import ResetParams, lib, ptr, stream_handle

pytestmark = pytest.mark.gpu


def _state(L, M, w):
    st = torch.zeros(L.reset_state_bytes(M, w), dtype=torch.uint8, device="cuda")
    assert L.reset_state_init(ptr(st), M, w, stream_handle()) == 0
    return st


def test_noalloc_matches_workspace_entry_on_two_calls():
    L = lib()
    M, V, w = 8, synth.LM_HEAD_VOCAB, 8
    params = ResetParams(0.6, 0.3, 1.0, w)
    st_ref, st_new = _state(L, M, w), _state(L, M, w)
    ws = torch.zeros(L.reset_workspace_bytes(M, V), dtype=torch.uint8, device="cuda")
    outs = {k: (torch.zeros(M, dtype=torch.int32, device="cuda"), torch.zeros(M, device="cuda"),
                torch.zeros(M, device="cuda")) for k in ("ref", "new")}
    starts = synth.reset_boundaries(2, M, p=0.5)
    us = synth.reset_uniforms(2, M, seed=11)
    for call, sigma in enumerate((3.0, 8.0)):
        logits = synth.reset_logits(call, M, V, sigma).cuda()
        st = torch.from_numpy(starts[call]).cuda()
        u = torch.from_numpy(us[call]).cuda()
        tok, H, T = outs["ref"]
        assert L.reset_sample(ptr(logits), M, V, ptr(st), ptr(u), ptr(st_ref), ctypes.byref(params), ptr(tok), ptr(H),
                              ptr(T), ptr(ws), ws.numel(), stream_handle()) == 0
        tok2, H2, T2 = outs["new"]
        assert L.reset_sample_noalloc(ptr(logits), M, V, ptr(st), ptr(u), ptr(st_new), ctypes.byref(params), ptr(tok2),
                                      ptr(H2), ptr(T2), stream_handle()) == 0
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), tok2.cpu().numpy()), call
        assert np.array_equal(T.cpu().numpy(), T2.cpu().numpy()), call
        h, h2 = H.cpu().numpy().astype(np.float64), H2.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(h - h2) <= 1e-4 * np.abs(h)), call


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = lib()
    M, w = 8, 8
    params = ResetParams(0.6, 0.3, 1.0, w)
    st = _state(L, M, w)
    small = torch.zeros((M, 64), device="cuda")          # never read: the call is rejected first
    tok = torch.zeros(M, dtype=torch.int32, device="cuda")
    u = torch.zeros(M, device="cuda")
    V = 2048 * 513                                        # 8 * 513 chunks > 4096
    rc = L.reset_sample_noalloc(ptr(small), M, V, None, ptr(u), ptr(st), ctypes.byref(params), ptr(tok), None, None,
                                stream_handle())
    assert rc == 2                                        # NVFP4_ERR_SHAPE


def _status(L):
    code = ctypes.c_uint(0)
    assert L.nvfp4_device_status(ctypes.byref(code)) == 0
    return code.value


def test_noalloc_across_shapes_and_top_p():
    """Calls of different shapes, with and without top-p, one after another on
    the shared static array (its layout depends on M and V, and its counters
    are cleared by each call): every call matches reset_sample on a fresh
    workspace, and no device error is recorded."""
    L = lib()
    w = 8
    _status(L)
    seq = [(8, synth.LM_HEAD_VOCAB, 1.0), (3, 2049, 0.9), (64, 4096, 0.95), (1, 1, 1.0),
           (8, synth.LM_HEAD_VOCAB, 0.95), (5, 70001, 1.0), (2, 300001, 0.95), (3, 2049, 0.9),
           (2, 300001, 1.0), (64, synth.LM_HEAD_VOCAB, 0.95)]
    for i, (M, V, top_p) in enumerate(seq):
        params = ResetParams(0.6, 0.3, 1.0, w, 0, top_p)
        st_ref, st_new = _state(L, M, w), _state(L, M, w)
        ws = torch.zeros(L.reset_workspace_bytes(M, V), dtype=torch.uint8, device="cuda")
        us = synth.reset_uniforms(2, M, seed=20 + i)
        for call in range(2):
            logits = synth.reset_logits(call + 10 * i, M, V, (1.0, 3.0, 8.0)[(i + call) % 3]).cuda()
            u = torch.from_numpy(us[call]).cuda()
            ref = [torch.zeros(M, dtype=torch.int32, device="cuda"), torch.zeros(M, device="cuda"),
                   torch.zeros(M, device="cuda")]
            new = [torch.zeros(M, dtype=torch.int32, device="cuda"), torch.zeros(M, device="cuda"),
                   torch.zeros(M, device="cuda")]
            assert L.reset_sample(ptr(logits), M, V, None, ptr(u), ptr(st_ref), ctypes.byref(params), ptr(ref[0]),
                                  ptr(ref[1]), ptr(ref[2]), ptr(ws), ws.numel(), stream_handle()) == 0
            assert L.reset_sample_noalloc(ptr(logits), M, V, None, ptr(u), ptr(st_new), ctypes.byref(params),
                                          ptr(new[0]), ptr(new[1]), ptr(new[2]), stream_handle()) == 0
            torch.cuda.synchronize()
            assert np.array_equal(ref[0].cpu().numpy(), new[0].cpu().numpy()), (M, V, top_p, call)
            assert np.array_equal(ref[2].cpu().numpy(), new[2].cpu().numpy()), (M, V, top_p, call)
            h, h2 = ref[1].cpu().numpy().astype(np.float64), new[1].cpu().numpy().astype(np.float64)
            assert np.all(np.abs(h - h2) <= 1e-4 * np.maximum(np.abs(h), 1e-6)), (M, V, top_p, call)
    assert _status(L) == 0
