"""The Python binding refuses, before any launch, what the kernels cannot
take: tensors in host memory (there is no CPU path: the product fails
loudly instead), wrong dtypes, and pools whose layout is not
[num_pages][Hkv][16][128] with [num_pages][Hkv][16] fp32 scales for INT8.
Runs without a GPU: the library loads and nothing is launched."""
import pytest
import torch

pk = pytest.importorskip("paged_kv_flash_gb300.pagedkv")


def i32(*v):
    return torch.tensor(v, dtype=torch.int32)


def bt():
    return i32(0, 1, 2, 3).view(1, 4)


def test_host_memory_pool_is_refused():
    for dtype in (torch.bfloat16, torch.int8):
        pool = pk.Pool.empty(4, 2, dtype=dtype, device="cpu")
        with pytest.raises(ValueError, match="pool.k"):
            pool.c()


def test_host_memory_inputs_are_refused():
    pool = pk.Pool.empty(4, 2, device="cpu")
    kn = torch.zeros((1, 2, 128), dtype=torch.bfloat16)
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pk.kv_append(pool, kn, kn, i32(0, 1), bt(), i32(1))
    with pytest.raises(ValueError):
        pk.paged_attn_decode(pool, q, bt(), i32(1), 1, 0.088)
    with pytest.raises(ValueError):
        pk.paged_attn_decode_noalloc(pool, q, bt(), i32(1), 1, 0.088)
    with pytest.raises(ValueError):
        pk.paged_attn_prefill(pool, q, i32(0, 1), bt(), i32(1), 1, 0.088,
                              workspace=torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError):
        pk.paged_attn_decode_multi(pool, q, i32(0, 1), bt(), i32(1), 1, 1, 0.088)


def _cuda_stub(monkeypatch):
    """Lets the layout checks run on host tensors: _need keeps its dtype and
    contiguity tests and drops the device test."""
    def need(t, dtype, name):
        if t.dtype != dtype or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous {dtype} tensor")
    monkeypatch.setattr(pk, "_need", need)


def test_pool_layout_checks(monkeypatch):
    _cuda_stub(monkeypatch)
    shape = (4, 2, 16, 128)
    bf = lambda s=shape: torch.zeros(s, dtype=torch.bfloat16)
    i8 = lambda s=shape: torch.zeros(s, dtype=torch.int8)
    f32 = lambda s=shape[:3]: torch.zeros(s, dtype=torch.float32)
    pk.Pool(bf(), bf())._validate()                        # well formed
    pk.Pool(i8(), i8(), f32(), f32())._validate()
    bad = [
        pk.Pool(bf((4, 2, 16, 64)), bf((4, 2, 16, 64))),      # head_dim
        pk.Pool(bf((4, 2, 8, 128)), bf((4, 2, 8, 128))),      # page size
        pk.Pool(bf(), bf((5, 2, 16, 128))),                   # k and v differ
        pk.Pool(bf(), i8()),                                  # mixed dtypes
        pk.Pool(bf(), bf(), f32(), f32()),                    # bf16 pool with scales
        pk.Pool(i8(), i8()),                                  # INT8 pool without scales
        pk.Pool(i8(), i8(), f32(), None),
        pk.Pool(i8(), i8(), f32((4, 2)), f32()),              # scale shape
        pk.Pool(i8(), i8(), f32().to(torch.float64), f32()),  # scale dtype
        pk.Pool(bf().transpose(0, 1), bf()),                  # not contiguous
    ]
    for p in bad:
        with pytest.raises(ValueError):
            p._validate()


def test_struct_is_rebuilt_and_rechecked_when_a_tensor_changes(monkeypatch):
    _cuda_stub(monkeypatch)
    pool = pk.Pool(torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16),
                   torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16))
    c1 = pool.c()
    assert pool.c() is c1                                  # cached while nothing changes
    pool.v = torch.zeros((4, 3, 16, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pool.c()
