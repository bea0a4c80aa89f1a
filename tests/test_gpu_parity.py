"""GPU parity of the CUDA path (through the C ABI) with the fp64 CPU oracle,
at sizes the oracle finishes in seconds that span several tiles and ragged
tails, plus the method's edge cases."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_cores, check_out
from sparse_long_context_cca_gb300 import api
from sparse_long_context_cca_gb300.inputs import make_qkv
from sparse_long_context_cca_gb300.workloads import TINY_F32, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "these tests need a GPU"
    api.load_library()


def wl(B, Hq, Hkv, N, d, g, w, dtype="bf16", seed=5, hh=0.01):
    return Workload(f"test B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} g{g} w{w} {dtype}", B, Hq, Hkv, N, d, g, w,
                    dtype, seed, hh)


POOL_CASES = [
    wl(1, 2, 2, 256, 128, 16, 1), wl(2, 4, 2, 512, 128, 8, 1), wl(1, 2, 2, 192, 128, 64, 1),
    wl(1, 1, 1, 96, 128, 1, 1), wl(1, 2, 2, 120, 128, 3, 1), wl(1, 4, 1, 256, 128, 32, 1),
    wl(1, 2, 2, 256, 64, 16, 1), wl(1, 2, 2, 320, 128, 40, 1),
    wl(1, 2, 2, 256, 64, 16, 1, "f32"), wl(1, 4, 2, 256, 128, 8, 1, "f32"), wl(1, 2, 2, 60, 64, 5, 1, "f32"),
]


@pytest.mark.parametrize("w", POOL_CASES, ids=lambda w: w.name)
def test_pool_parity(w):
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    torch.cuda.synchronize()
    Kr, Vr = oracle.pool(Q, K, V, w.g)
    check_cores(Kc, Vc, Kr, Vr, Q.dtype, w.name)


ATTN_CASES = [
    TINY_F32,
    wl(1, 2, 2, 512, 64, 8, 100, "f32"),
    wl(2, 4, 2, 384, 128, 16, 64, "f32"),
    wl(1, 2, 2, 256, 128, 16, 32),          # tiny shape in bf16
    wl(1, 2, 2, 1008, 128, 16, 160),        # ragged last query tile (1008 = 7*128 + 112)
    wl(1, 2, 2, 384, 128, 16, 512),         # w >= N: causal attention, no cores
    wl(1, 2, 2, 256, 128, 4, 1),            # w = 1: one local key per row
    wl(1, 2, 2, 384, 128, 1, 64),           # g = 1: equal to causal attention
    wl(1, 2, 2, 2048, 128, 64, 256),
    wl(1, 8, 2, 1024, 128, 16, 128),        # GQA, r = 4
    wl(2, 2, 2, 640, 128, 8, 96),           # B = 2, w not a multiple of the tile
    wl(1, 2, 2, 4096, 128, 8, 256),         # several core tiles per query tile
    wl(1, 2, 1, 1920, 128, 24, 300),        # g not a power of two, GQA r = 2
    wl(1, 1, 1, 16, 128, 16, 4),            # a single group, N far below one tile
]


@pytest.mark.parametrize("w", ATTN_CASES, ids=lambda w: w.name)
def test_prefill_parity(w):
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w)
    torch.cuda.synchronize()
    Or, Lr, Kr, Vr = oracle.prefill(Q, K, V, w.g, w.w)
    check_cores(Kc, Vc, Kr, Vr, Q.dtype, w.name)
    check_out(O, LSE, Or, Lr, Q.dtype, w.name + " end-to-end")
    # attention alone, fed the GPU's own core tokens
    Oa, La = oracle.attn(Q, K, V, Kc, Vc, w.g, w.w)
    check_out(O, LSE, Oa, La, Q.dtype, w.name + " attention-only")


@pytest.mark.parametrize("w", [wl(1, 2, 2, 1024, 128, 16, 128), wl(1, 2, 2, 512, 64, 16, 64, "f32")],
                         ids=lambda w: w.name)
def test_repeatable_bitwise(w):
    """Two runs on the same inputs give identical bits (no races)."""
    Q, K, V = make_qkv(w, "cuda")
    a = api.cca_prefill(Q, K, V, w.g, w.w)
    b = api.cca_prefill(Q, K, V, w.g, w.w)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_scale_argument():
    w = wl(1, 2, 2, 512, 128, 16, 64)
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, scale=0.05)
    torch.cuda.synchronize()
    Or, Lr, Kr, Vr = oracle.prefill(Q, K, V, w.g, w.w, scale=0.05)
    check_out(O, LSE, Or, Lr, Q.dtype, "scale=0.05")


def test_streams_and_preallocated_outputs():
    w = wl(1, 4, 4, 768, 128, 16, 128)
    Q, K, V = make_qkv(w, "cuda")
    s = torch.cuda.Stream()
    out = (torch.full_like(Q, float("nan")), torch.full((1, 4, 768), float("nan"), device="cuda"),
           torch.empty(1, 4, 48, 128, dtype=Q.dtype, device="cuda"),
           torch.empty(1, 4, 48, 128, dtype=Q.dtype, device="cuda"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        api.cca_prefill(Q, K, V, w.g, w.w, out=out, stream=s)
    s.synchronize()
    Or, Lr, _, _ = oracle.prefill(Q, K, V, w.g, w.w)
    check_out(out[0], out[1], Or, Lr, Q.dtype, "side stream")


def test_dev_status_stays_zero():
    w = wl(1, 2, 2, 512, 128, 16, 64)
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.cca_attn_fwd(Q, K, V, Kc, Vc, w.g, w.w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_causal_attention_comparator():
    """The full-attention comparator (same kernel, g = 1, w = N) is causal attention."""
    w = wl(1, 4, 2, 1000, 128, 1, 1000)
    Q, K, V = make_qkv(w, "cuda")
    O, LSE = api.causal_attention(Q, K, V)
    torch.cuda.synchronize()
    Or, Lr, _, _ = oracle.prefill(Q, K, V, 1, w.N)
    check_out(O, LSE, Or, Lr, Q.dtype, "causal comparator")


VARIANT_CASES = [
    (wl(1, 4, 2, 1024, 128, 16, 200), 1, 0), (wl(1, 4, 2, 1024, 128, 16, 200), 2, 0),
    (wl(1, 4, 2, 1024, 128, 16, 200), 0, 1), (wl(2, 2, 2, 1536, 128, 8, 333), 2, 1),
    (wl(1, 2, 2, 512, 64, 16, 70, "f32"), 1, 1), (wl(1, 2, 1, 512, 128, 8, 100, "f32"), 2, 0),
    (wl(1, 2, 2, 384, 128, 1, 64), 0, 1),
]


@pytest.mark.parametrize("w,pool_mode,window_mode", VARIANT_CASES,
                         ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_variants_parity(w, pool_mode, window_mode):
    """Mean / max pooling and the group-aligned window (the pages' ablations)."""
    Q, K, V = make_qkv(w, "cuda")
    O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    torch.cuda.synchronize()
    Or, Lr, Kr, Vr = oracle.prefill(Q, K, V, w.g, w.w, pool_mode=pool_mode, window_mode=window_mode)
    check_cores(Kc, Vc, Kr, Vr, Q.dtype, f"{w.name} pool {pool_mode}")
    check_out(O, LSE, Or, Lr, Q.dtype, f"{w.name} pool {pool_mode} window {window_mode}")


def test_output_alignment_16_bytes():
    """O only 16-byte aligned (the ABI minimum) takes the epilogue's 16-byte stores and gives
    the same bits as a 32-byte-aligned O."""
    w = wl(1, 2, 2, 384, 128, 16, 100)
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g)
    O1, L1 = api.cca_attn_fwd(Q, K, V, Kc, Vc, w.g, w.w)
    buf = torch.empty(Q.numel() + 16, dtype=Q.dtype, device="cuda")
    assert buf.data_ptr() % 32 == 0
    O2 = buf[8:8 + Q.numel()].view(Q.shape)  # 16 bytes past a 32-byte boundary
    assert O2.data_ptr() % 32 == 16
    O2, L2 = api.cca_attn_fwd(Q, K, V, Kc, Vc, w.g, w.w, O=O2)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


# Pooling of small groups: g of 1, 2 or 4 row passes takes the kernel that packs several
# whole groups into one chunk (per dtype and d: bf16 d128 g 2/4/8, bf16 d64 g 4/8/16,
# f32 d128 g 1/2/4, f32 d64 g 2/4/8).  Group counts are not multiples of the groups per
# chunk, so the last chunk of every (batch, KV head) is ragged.
SMALL_GROUP_CASES = [
    (wl(1, 2, 2, 2 * 101, 128, 2, 40), 0), (wl(2, 4, 2, 4 * 37, 128, 4, 30), 1),
    (wl(1, 8, 2, 8 * 45, 128, 8, 60), 0), (wl(1, 4, 4, 8 * 29, 128, 8, 60), 2),
    (wl(1, 4, 1, 4 * 50, 64, 4, 40), 0), (wl(1, 2, 2, 8 * 33, 64, 8, 50), 2),
    (wl(2, 2, 1, 16 * 21, 64, 16, 64), 1),
    (wl(1, 2, 2, 77, 128, 1, 20, "f32"), 0), (wl(1, 4, 2, 2 * 61, 128, 2, 20, "f32"), 2),
    (wl(1, 2, 2, 4 * 19, 128, 4, 20, "f32"), 1),
    (wl(1, 2, 2, 2 * 45, 64, 2, 20, "f32"), 0), (wl(1, 4, 2, 4 * 27, 64, 4, 20, "f32"), 0),
    (wl(1, 2, 1, 8 * 23, 64, 8, 20, "f32"), 2),
]


@pytest.mark.parametrize("w,pool_mode", SMALL_GROUP_CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_small_group_pooling(w, pool_mode):
    Q, K, V = make_qkv(w, "cuda")
    Kc, Vc = api.cca_pool(Q, K, V, w.g, pool_mode=pool_mode)
    torch.cuda.synchronize()
    Kr, Vr = oracle.pool(Q, K, V, w.g, pool_mode=pool_mode)
    check_cores(Kc, Vc, Kr, Vr, Q.dtype, f"{w.name} pool {pool_mode}")
    if pool_mode == 0 and (w.d == 128 or w.dtype == "f32"):
        O, LSE = api.cca_attn_fwd(Q, K, V, Kc, Vc, w.g, w.w)
        torch.cuda.synchronize()
        Or, Lr = oracle.attn(Q, K, V, Kr, Vr, w.g, w.w)
        check_out(O, LSE, Or, Lr, Q.dtype, f"{w.name} prefill")


def test_concurrent_host_threads():
    """Two host threads call the library at once, each on its own stream with its own inputs
    (prefill, decode, backward): the per-device state the library keeps (launch attributes,
    occupancy, cluster size) is set up under a lock, and every call builds its own tensor maps
    and parameters, so the results equal the same calls made one after another."""
    import threading

    shapes = [wl(1, 4, 2, 1024, 128, 16, 200, seed=101), wl(1, 2, 2, 1536, 128, 32, 300, seed=102)]
    inputs = [make_qkv(w, "cuda") for w in shapes]
    torch.cuda.synchronize()  # the inputs are made on the default stream

    def run(k, out, stream):
        w = shapes[k]
        Q, K, V = inputs[k]
        with torch.cuda.stream(stream):
            for _ in range(4):
                O, LSE, Kc, Vc = api.cca_prefill(Q, K, V, w.g, w.w, stream=stream)
                pos = w.N - 1
                Od, Ld = api.cca_decode_fwd(Q[:, :, pos].contiguous(), K, V, Kc, Vc, pos, w.g, w.w, stream=stream)
                dQ, dK, dV = api.cca_prefill_bwd(Q, K, V, Kc, Vc, O, LSE, torch.ones_like(O), w.g, w.w,
                                                 stream=stream)
            stream.synchronize()
        out[k] = (O, LSE, Od, Ld, dQ, dK, dV)

    ref = [None, None]
    for k in range(2):
        run(k, ref, torch.cuda.Stream())
    got = [None, None]
    threads = [threading.Thread(target=run, args=(k, got, torch.cuda.Stream())) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for k in range(2):
        for a, b in zip(got[k], ref[k]):
            assert torch.equal(a, b), k
