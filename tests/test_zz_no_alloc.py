"""tk_decode_noalloc: decoding for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: a server whose memory pool already holds
the device's memory, or a latency-critical path that must not enter the
allocator. tk_decode_noalloc serves them with a fixed scratch array compiled
into the library instead of a workspace. These tests call it through the C ABI
and compare its bytes with tk_decode's (the workspace entry point), exactly,
on two calls in a row. This file is collected last on purpose.
"""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gpu_tok(full_table):
    import byte_level_bpe_gb300 as tk
    t = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 22, max_segments=64)
    yield t
    t.close()


def _noalloc(tok, d_ids, cap):
    from byte_level_bpe_gb300 import native
    out = torch.empty(max(cap, 1), dtype=torch.uint8, device="cuda")
    rc, m = native.tk_decode_noalloc(tok.handle, d_ids.data_ptr() if d_ids.numel() else None,
                                     d_ids.numel(), out.data_ptr(), cap,
                                     torch.cuda.current_stream().cuda_stream, raise_on_error=False)
    return rc, m, out


def test_matches_workspace_decode_two_calls(gpu_tok, full_table):
    from byte_level_bpe_gb300 import native
    big = workloads.prose_text(full_table, 1 << 20, seed=41) + "<|endoftext|> 中文 \U0001F600".encode()
    small = workloads.prose_text(full_table, 5000, seed=42)
    ids_big, _ = gpu_tok.encode_segments([(big, True)])
    ids_small, _ = gpu_tok.encode_segments([(small, False)])
    assert ids_big.numel() > 2048 * 4  # several tiles of the decode kernel
    for ids in (ids_big, ids_small, ids_big):  # two (and three) calls in a row
        ref = gpu_tok.decode_device(ids).cpu().numpy().tobytes()
        rc, m, out = _noalloc(gpu_tok, ids, len(ref))
        assert rc == native.TK_OK, native.load().tk_last_error()
        assert m == len(ref)
        assert out[:m].cpu().numpy().tobytes() == ref


def test_errors(gpu_tok):
    from byte_level_bpe_gb300 import native
    ids = torch.tensor([65, 66, 100256, 67], dtype=torch.int32, device="cuda")  # 100256: reserved gap
    rc, _, _ = _noalloc(gpu_tok, ids, 64)
    assert rc == native.TK_E_BADID
    assert b"index 2" in native.load().tk_last_error()
    ids = torch.tensor([65, 66, 67], dtype=torch.int32, device="cuda")
    rc, m, _ = _noalloc(gpu_tok, ids, 2)
    assert rc == native.TK_E_CAPACITY and m == 3
    too_many = torch.zeros((1 << 20) + 1, dtype=torch.int32, device="cuda")
    rc, _, _ = _noalloc(gpu_tok, too_many, 16)
    assert rc == native.TK_E_LIMIT
    rc, m, out = _noalloc(gpu_tok, ids, 16)  # usable again after the errors
    assert rc == native.TK_OK and out[:m].cpu().numpy().tobytes() == b"ABC"


def test_exact_limit(gpu_tok, full_table):
    """The largest call the fixed scratch takes (1,048,576 ids: its look-back
    descriptors used to the last one) and one that ends in a partial tile,
    each with multi-byte ids, against tk_decode."""
    from byte_level_bpe_gb300 import native
    ids_cjk, _ = gpu_tok.encode_segments([("中文 \U0001F600 don't", False)])
    pattern = ids_cjk.repeat((1 << 20) // ids_cjk.numel() + 1)
    for n in (1 << 20, (1 << 20) - 2047):
        ids = pattern[:n].contiguous()
        ref = gpu_tok.decode_device(ids).cpu().numpy().tobytes()
        for _ in range(2):
            rc, m, out = _noalloc(gpu_tok, ids, len(ref))
            assert rc == native.TK_OK, native.load().tk_last_error()
            assert m == len(ref)
            assert out[:m].cpu().numpy().tobytes() == ref
