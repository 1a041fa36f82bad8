"""The sampling-verification entry point that allocates nothing.

Callers that cannot allocate device memory (a framework that owns every
allocation, a plugin in another runtime, a serving loop that must not call
the allocator while running) use dflash_verify_sample_noalloc, whose scratch
is an array inside the library. Its results must equal the workspace
variant's, on two calls in a row (the array keeps the previous call's
contents, which must not leak into the next). This file is collected last.
"""
import ctypes as C

import pytest
import torch

import synthetic_inputs as SI

pytestmark = pytest.mark.gpu


def _inputs(S, V, seed):
    tl = SI.make_logits((S, 16, V), 2.0, seed, device="cuda")
    dl = (tl[:, :15].float() + 0.4 * SI.make_logits((S, 15, V), 1.0, seed + 1, device="cuda").float()).to(
        torch.bfloat16
    )
    g = torch.Generator(device="cuda").manual_seed(seed + 2)
    draft = torch.multinomial(torch.softmax(dl.float(), -1).view(-1, V), 1, generator=g).view(S, 15).to(torch.int32)
    u = SI.make_uniforms((S, 16, 2), seed + 3, device="cuda")
    return draft.contiguous(), tl, dl, u


def test_noalloc_sampling_verify_equals_workspace_variant():
    import block_diffusion_speculative_tap_gb300 as D
    from block_diffusion_speculative_tap_gb300 import _abi as A

    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (S, V, T) in enumerate([(12, 151936, 1.0), (5, 4096, 0.8)]):
        draft, tl, dl, u = _inputs(S, V, 100 + call)
        a_ref, t_ref = D.verify_sample(draft, tl, dl, u, T)
        acc = torch.full((S,), -7, dtype=torch.int32, device="cuda")
        toks = torch.full((S, 16), -7, dtype=torch.int32, device="cuda")
        rc = A.lib.dflash_verify_sample_noalloc(
            S, V, C.c_void_p(draft.data_ptr()), 1, C.c_void_p(tl.data_ptr()), C.c_void_p(dl.data_ptr()),
            C.c_void_p(u.data_ptr()), T, C.c_void_p(acc.data_ptr()), C.c_void_p(toks.data_ptr()), stream,
        )
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert torch.equal(acc, a_ref), call
        assert torch.equal(toks, t_ref), call


def test_noalloc_rejects_more_streams_than_its_array_holds():
    from block_diffusion_speculative_tap_gb300 import _abi as A

    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    lg = torch.zeros(16, 8, dtype=torch.bfloat16, device="cuda")
    rc = A.lib.dflash_verify_sample_noalloc(
        1025, 8, C.c_void_p(x.data_ptr()), 1, C.c_void_p(lg.data_ptr()), C.c_void_p(lg.data_ptr()),
        C.c_void_p(lg.data_ptr()), 1.0, C.c_void_p(x.data_ptr()), C.c_void_p(x.data_ptr()), stream,
    )
    assert rc == A.E_WORKSPACE
