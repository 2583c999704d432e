"""paged_attn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (code inside an allocator or memory-pool callback, serving
loops that must not block on the allocator or fail with out-of-memory mid-step,
hosts that only hold their own input and output buffers).  Its chunk partials
live in a fixed array inside the library, so the caller passes no workspace.

This file is collected last on purpose: if the GPU test here fails, a run that
stops at the first failure has already run every other test.  It must pass both
alone in a fresh process and after the other tests (the shared array then holds
whatever an earlier call left in it)."""
import numpy as np
import pytest
import torch

from attn_fwd_02_gb300 import workloads

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3  # the parity tolerances of the other GPU tests
SCRATCH_LIMIT = 7  # ATTN_ERR_SCRATCH_LIMIT


def _both(binding, shape, ctx):
    inp = workloads.decode_inputs(shape, ctx_lens=ctx)
    d = {k: v.cuda() for k, v in inp.items()}
    o_ref, lse_ref = binding.paged_attn_decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"],
                                               d["ctx_lens"], shape.scale)
    o = torch.full_like(d["q"], float("nan"))
    lse = torch.full(d["q"].shape[:2], float("nan"), device="cuda")
    binding.paged_attn_decode_noalloc(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["ctx_lens"],
                                      shape.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.attn_check_device_status() == 0
    err = (o.float() - o_ref.float()).abs()
    assert torch.isfinite(o).all()
    assert err.max().item() <= O_MAX and err.mean().item() <= O_MEAN
    inf = torch.isneginf(lse_ref)
    assert torch.equal(torch.isneginf(lse), inf)
    if (~inf).any():
        assert (lse[~inf] - lse_ref[~inf]).abs().max().item() <= LSE_MAX
    # and on its own against the fp64 oracle, within the same tolerances
    from oracle import oracle
    o64, lse64 = oracle.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"],
                                     shape.scale)
    err64 = np.abs(o.float().cpu().numpy() - o64)
    assert err64.max() <= O_MAX and err64.mean() <= O_MEAN
    lse_c = lse.cpu().numpy()
    fin = np.isfinite(lse64)
    assert np.array_equal(np.isneginf(lse_c), np.isneginf(lse64))
    if fin.any():
        assert np.abs(lse_c[fin] - lse64[fin]).max() <= LSE_MAX


@pytest.mark.gpu
def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attn_fwd_02_gb300 import binding, build
    build.build()
    # first call: multi-chunk contexts; second call: different sizes, so the shared
    # array holds the first call's partials when the second one starts
    _both(binding, workloads.DecodeShape("noalloc call 1", 4, 8, 128, (1, 3000), seed=90), [3000, 1, 513, 2048])
    _both(binding, workloads.DecodeShape("noalloc call 2", 6, 4, 64, (1, 1200), seed=91),
          [700, 0, 1200, 16, 17, 511])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # host-side check, before any device work: 64 x 64 heads of 8192-token contexts at d=128
    # need 64*64*16*(128+4)*4 bytes = 34.6 MB of partials, more than the 12 MiB array
    from attn_fwd_02_gb300 import binding, build
    build.build()
    lib = binding.load_library()
    a = 1 << 20
    st = lib.paged_attn_decode_noalloc(a, a, a, a, a, 16, a, None, 64, 64, 128, 512, 10, 0.1, None)
    assert st == SCRATCH_LIMIT
    assert "12 MiB" in binding.attn_status_string(st)
    # the workload of the benchmark (32 x 32 heads, 512 pages) fits
    assert lib.paged_attn_decode_workspace_size(32, 32, 128, 512, 16) <= 12 << 20
