"""GPU tests of the write-back host offload and prefetch of checkpoint objects: the host copy
is the object's bytes, a prefetch puts them back bit for bit into fresh pages, and a decode
step continues from a prefetched checkpoint exactly as from the original."""
import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads
from oracle import policy

from kda_cases import random_state, read_object_bytes, write_object

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype,d,H,page_bytes", [("bf16", 128, 32, 65536), ("f32", 64, 3, 4096),
                                                  ("bf16", 128, 5, 768)])
def test_offload_and_prefetch_are_byte_copies(dtype, d, H, page_bytes):
    dt = kda.DTYPES[dtype]
    n = 3
    P = policy.object_pages(H, d, dtype, page_bytes)
    nb = policy.object_bytes(H, d, dtype)
    pool = kda.Pool(page_bytes, 2 * n * P + 8, DEV)
    src = kda.kda_page_alloc(pool, n * P).reshape(n, P)
    g = torch.Generator(device=DEV).manual_seed(4)
    for p in src.reshape(-1):
        pool.page_view(int(p)).copy_(torch.randint(0, 256, (page_bytes,), generator=g, device=DEV,
                                                   dtype=torch.int32).to(torch.uint8))
    host = torch.zeros(n * nb, dtype=torch.uint8).pin_memory()
    ws = torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_ckpt_offload(pool, H, d, dt, src.reshape(-1), host, ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    hb = host.numpy().tobytes()
    for i in range(n):
        assert hb[i * nb:(i + 1) * nb] == read_object_bytes(pool, src[i], nb)
    # evict, then prefetch into fresh pages
    kda.kda_page_decref(pool, src.reshape(-1))
    back = kda.kda_ckpt_prefetch(pool, H, d, dt, n, host, ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    assert back.shape == (n, P)
    for i in range(n):
        assert read_object_bytes(pool, back[i], nb) == hb[i * nb:(i + 1) * nb]


def test_decode_continues_from_a_prefetched_checkpoint():
    dtype, d, H, B = "bf16", 128, 4, 3
    dt = kda.DTYPES[dtype]
    page_bytes = 65536
    P = policy.object_pages(H, d, dtype, page_bytes)
    nb = policy.object_bytes(H, d, dtype)
    pool = kda.Pool(page_bytes, 6 * B * P + 8, DEV)
    ck = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    gen = torch.Generator().manual_seed(12)
    for b in range(B):
        S, W = random_state(H, d, dtype, gen)
        write_object(pool, ck[b], S, W, dtype)
    ws = torch.empty(kda.kda_copy_workspace_bytes(B, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    # path 1: restore the resident checkpoint
    a1 = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    kda.kda_ckpt_restore(pool, H, d, dt, ck.reshape(-1), a1.reshape(-1), ws, st)
    # path 2: offload, evict, prefetch, restore
    host = torch.zeros(B * nb, dtype=torch.uint8).pin_memory()
    kda.kda_ckpt_offload(pool, H, d, dt, ck.reshape(-1), host, ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    kda.kda_ckpt_release(pool, ck.reshape(-1), P)
    kda.kda_page_decref(pool, ck.reshape(-1))
    back = kda.kda_ckpt_prefetch(pool, H, d, dt, B, host, ws, st)
    a2 = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    kda.kda_ckpt_restore(pool, H, d, dt, back.reshape(-1), a2.reshape(-1), ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    kda.kda_ckpt_release(pool, back.reshape(-1), P)
    conv_w = (torch.randn(H, 3 * d, 4, generator=gen) * 0.5).to(DEV)
    t = workloads.decode_step_tokens(B, H, d, dtype, 12, 0, DEV)
    outs = []
    for act in (a1, a2):
        o = torch.empty_like(t["q"])
        kda.kda_decode_step(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, o,
                            torch.from_numpy(act).to(DEV), st)
        assert kda.kda_sync_status(st)[0] == kda.KDA_OK
        outs.append(o)
    assert torch.equal(outs[0], outs[1])
    for b in range(B):
        assert read_object_bytes(pool, a1[b], nb) == read_object_bytes(pool, a2[b], nb)
