"""Host-side failure paths on a GPU, none of which faults, traps or hangs it.

* hs_wait_offload: a bounded host-side wait for an offload's copy event.  The
  copy is held back by a host-side gate -- a host function queued on the side
  stream ahead of the offload blocks (on the host) until the test opens it --
  so the event is not complete and the wait must give up with HS_ERR_TIMEOUT;
  once the gate opens, the wait returns HS_OK and the host rows hold the page.
  Page "GLM 5.3 Optimizations, Part 1", section "How it works": the CPU copy
  serves prefix reuse once the transfer completes.
* hs_pool_create failing part way (a device allocation after the pinned host
  pool does not fit) returns HS_ERR_OOM and leaves nothing allocated.
"""
import ctypes
import os
import threading

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402


def _cudart():
    """The CUDA runtime this process already uses (torch's), else the toolkit's."""
    torch.cuda.init()
    with open("/proc/self/maps") as f:
        for line in f:
            path = line.split()[-1]
            if "libcudart.so" in os.path.basename(path):
                return ctypes.CDLL(path)
    for cand in ("libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return ctypes.CDLL(cand)
        except OSError:
            pass
    pytest.skip("no CUDA runtime library to queue a host function with")


HOSTFN = ctypes.CFUNCTYPE(None, ctypes.c_void_p)


def test_wait_offload_times_out_while_a_host_gate_holds_the_copy():
    rt = _cudart()
    rt.cudaLaunchHostFunc.argtypes = [ctypes.c_void_p, HOSTFN, ctypes.c_void_p]
    rt.cudaLaunchHostFunc.restype = ctypes.c_int
    R, L, K, B, P = 2, 2, 64, 256, 256
    pool = hs.Pool(R, L, K, B, P, 576, 8, 8 * P * R, 8)
    hs.hs_set_request(pool.handle, 1, 4 * P, 8 * P)
    blk = pool.hot_blocks + 3  # a resident block
    rows = np.stack([synth.rows(21, 1, l, 2 * P, P) for l in range(L)])
    for l in range(L):
        pool.kv_pool[l, blk * P:(blk + 1) * P].copy_(torch.from_numpy(rows[l].view(np.int16)))
    hs.hs_map_page(pool.handle, 1, 2, blk)
    pool.host_pool[:, 8 * P + 2 * P:8 * P + 3 * P] = 0
    torch.cuda.synchronize()

    gate = threading.Event()
    entered = threading.Event()

    def hold(_):
        entered.set()
        gate.wait(20.0)  # bounded: never holds the stream past 20 s

    cb = HOSTFN(hold)
    # streams of their own (the legacy default stream would wait for the gate
    # itself), and an event that exists before the gate closes
    side = torch.cuda.Stream()
    main = torch.cuda.Stream()
    done = torch.cuda.Event()
    # one offload with the gate open first: the copy kernel's first launch may
    # load its module, which would wait for a blocked host function
    hs.hs_offload_prefix(pool.handle, 1, 2, main, side, done)
    assert hs.hs_wait_offload(done, 10_000_000_000) == hs.HS_OK
    pool.host_pool[:, 8 * P + 2 * P:8 * P + 3 * P] = 0
    assert rt.cudaLaunchHostFunc(side.cuda_stream, cb, None) == 0
    hs.hs_offload_prefix(pool.handle, 1, 2, main, side, done)
    try:
        assert entered.wait(10.0)
        assert hs.hs_wait_offload(done, 50_000_000) == hs.HS_ERR_TIMEOUT  # 50 ms
        assert hs.hs_wait_offload(done, 0) == hs.HS_ERR_TIMEOUT
        assert not np.any(pool.host_pool[:, 8 * P + 2 * P:8 * P + 3 * P])  # not copied yet
    finally:
        gate.set()
    assert hs.hs_wait_offload(done, 10_000_000_000) == hs.HS_OK
    got = np.asarray(pool.host_pool[:, 8 * P + 2 * P:8 * P + 3 * P]).view(np.uint16)
    assert np.array_equal(got, rows)
    torch.cuda.synchronize()
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()


def test_pool_create_failing_part_way_frees_what_it_allocated():
    """Device memory is squeezed so that the pool's position -> slot array
    (L x host_tokens int32, allocated after the pinned host pool) cannot be
    placed: HS_ERR_OOM, and the free device memory is what it was before."""
    warm = hs.Pool(1, 1, 64, 256, 256, 576, 16, 4096, 4)  # every kernel module loaded
    warm.close()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free0, _ = torch.cuda.mem_get_info()
    host_tokens = 1 << 28  # 16-byte rows: 4 GiB pinned host pool; 1 GiB index array
    leave = 768 << 20
    hold = torch.empty(free0 - leave, dtype=torch.uint8, device="cuda")
    try:
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 < (1 << 30)
        lib = hs.load()
        desc = hs.hs_pool_desc(1, 1, 64, 256, 256, 8, 16, 0, host_tokens, 4)
        out = ctypes.c_void_p(None)
        st = lib.hs_pool_create(ctypes.byref(desc), ctypes.byref(out))
        assert st == hs.HS_ERR_OOM and out.value is None
        free2, _ = torch.cuda.mem_get_info()
        assert abs(free2 - free1) < (8 << 20), (free1, free2)
    finally:
        del hold
        torch.cuda.empty_cache()
    # and a pool fits again afterwards
    pool = hs.Pool(1, 1, 64, 256, 256, 576, 16, 4096, 4)
    pool.close()


def test_host_pool_is_placed_on_the_devices_numa_node():
    """On a machine with several host NUMA nodes the pinned host pool sits on
    the node nearest the device (the PCI device's numa_node); with one node it
    is not placed (-1).  It is readable and writable from both sides either
    way."""
    pool = hs.Pool(1, 1, 64, 256, 256, 576, 16, 4096, 4)
    node = hs.hs_pool_host_numa_node(pool.handle)
    nodes = [d for d in os.listdir("/sys/devices/system/node")
             if d.startswith("node") and d[4:].isdigit()] if os.path.isdir(
                 "/sys/devices/system/node") else []
    bus = torch.cuda.get_device_properties(0)
    want = None
    pci = getattr(bus, "pci_bus_id", None)
    dom = getattr(bus, "pci_domain_id", 0)
    dev = getattr(bus, "pci_device_id", None)
    if pci is not None and dev is not None:
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/numa_node" % (dom, pci, dev)
        if os.path.exists(path):
            want = int(open(path).read().strip())
    if len(nodes) <= 1:
        assert node == -1
    elif want is not None and want >= 0:
        assert node == want, (node, want)
    else:
        assert node >= -1
    rows = synth.rows(3, 0, 0, 0, 256)
    pool.host_pool[0, :256] = rows
    d = torch.empty((256, 576), dtype=torch.int16, device="cuda")
    hs.hs_host_read(pool.raw.host_pool_device, 256 * 1152, d)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy().view(np.uint16), rows)
    pool.close()
