"""sub_verify_accept_static, the accept step for callers that cannot allocate
device memory while they decode: a runtime that owns the device's memory
through its own allocator and forbids libraries to call cudaMalloc or
cudaMallocAsync, or a decode loop that must not stall or fail on an
allocation once it has started.  The entry point uses a fixed scratch array
the library holds on each device instead.  It must give exactly what
sub_verify_accept gives, on two calls in a row (the second call reuses the
scratch the first one left), and it must take no memory from the device's
memory pool."""
import ctypes as C

import numpy as np
import pytest
import torch

import synthetic

DEV = "cuda"


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


def test_static_scratch_bound_is_checked_on_the_host(sub):
    # 40001 nodes need 40001 * 8 + 64 + 40001 * 4 bytes (no choice array
    # given): beyond the fixed scratch, rejected before any CUDA call
    t = sub.Tree()
    t.width, t.max_depth = 4, 10000
    fake = C.c_void_p(256)
    r = sub._verify_accept_static(fake, C.byref(t), 40001, 1024, 0, 1.0, 0, 0, fake, fake, fake,
                                  None, None)
    assert r == sub.SUB_EINVAL
    assert b"static accept scratch" in sub._lib.sub_last_error()


def _case(sub, mode, vocab, depth, width, seed):
    tok, par, dep = synthetic.random_tree(depth, width, seed, vocab)
    n = len(par)
    rng = np.random.default_rng(seed + vocab)
    lg = (rng.standard_normal((n, vocab)) * 3).astype(np.float32)
    # a matching chain along the root path of a deepest node
    path = [n - 1]
    while par[path[-1]] >= 0:
        path.append(int(par[path[-1]]))
    path = path[::-1]
    for u, c in zip(path[:-1], path[1:]):
        lg[u, tok[c]] = lg[u].max() + (5.0 if mode == 0 else 40.0)
    tr = sub.DeviceTree(depth, width, DEV)
    tr.token.copy_(tok)
    tr.parent.copy_(par)
    tr.depth.copy_(dep)
    return torch.tensor(lg, device=DEV), tr, n


@pytest.mark.gpu
@pytest.mark.parametrize("mode,vocab,depth,width", [(0, 152064, 48, 8), (1, 152064, 48, 8),
                                                    (0, 1024, 6, 3), (1, 5000, 3, 16)])
@pytest.mark.parametrize("with_choice", [True, False])
def test_static_matches_allocating_accept_twice(sub, mode, vocab, depth, width, with_choice):
    logits, tr, n = _case(sub, mode, vocab, depth, width, seed=mode + depth)
    kw = dict(mode=mode, temperature=0.6, seed=11, root_pos=301, with_choice=with_choice)
    ref = sub.verify_accept(logits, tr, n, **kw)
    torch.cuda.synchronize()
    for _ in range(2):
        got = sub.verify_accept_static(logits, tr, n, **kw)
        torch.cuda.synchronize()
        a = int(ref[1].item())
        assert a >= 1 and int(got[1].item()) == a
        assert torch.equal(got[0][:a], ref[0][:a])
        assert torch.equal(got[2], ref[2])
        if with_choice:
            assert torch.equal(got[3], ref[3])
        else:
            assert got[3] is None


def _default_pool_high_water():
    """Reset, then read back, the high-water mark of the device's default
    memory pool (the pool cudaMallocAsync draws from), through the CUDA driver API."""
    drv = C.CDLL("libcuda.so.1")
    dev = C.c_int()
    assert drv.cuDeviceGet(C.byref(dev), torch.cuda.current_device()) == 0
    pool = C.c_void_p()
    assert drv.cuDeviceGetDefaultMemPool(C.byref(pool), dev) == 0
    used_high = 8   # CU_MEMPOOL_ATTR_USED_MEM_HIGH

    def reset():
        zero = C.c_uint64(0)
        assert drv.cuMemPoolSetAttribute(pool, used_high, C.byref(zero)) == 0

    def read():
        v = C.c_uint64()
        assert drv.cuMemPoolGetAttribute(pool, used_high, C.byref(v)) == 0
        return v.value
    return reset, read


@pytest.mark.gpu
def test_static_accept_allocates_nothing(sub):
    """For callers that cannot allocate inside their decode loop: the static
    entry point draws no device memory, while the allocating one does (the
    control shows the measurement sees its per-call scratch)."""
    logits, tr, n = _case(sub, 0, 152064, 48, 8, seed=5)
    out = sub.verify_accept_static(logits, tr, n, root_pos=9)   # first call: set-up
    torch.cuda.synchronize()
    reset, read = _default_pool_high_water()
    reset()
    base = read()
    for _ in range(2):
        sub.verify_accept_static(logits, tr, n, root_pos=9, out=out)
    torch.cuda.synchronize()
    assert read() == base
    sub.verify_accept(logits, tr, n, root_pos=9)
    torch.cuda.synchronize()
    assert read() > base
