"""Thin Python binding of the C-ABI library libllar.so (include/llar.h).

Argument marshalling only: tensors become device pointers, names become
enum values, torch's current stream becomes the cudaStream_t. Every step of
the AllReduce runs in the library's CUDA kernels. There is no fallback: if
libllar.so is missing or a call fails, an exception is raised.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# LLAR_LIBRARY selects another build of the same sources (tuning variants)
LIB_PATH = os.environ.get("LLAR_LIBRARY") or os.path.join(HERE, "libllar.so")

DTYPES = {"fp32": 0, "fp16": 1, "bf16": 2}
PROTOCOLS = {"auto": 0, "ll": 1, "sentinel": 2, "ll128": 3,
             "fixed_oneshot": 4, "fixed_twoshot": 5, "ll128_direct": 6}
PROTOCOL_NAMES = {v: k for k, v in PROTOCOLS.items()}
INJECT = {"none": 0, "skip": 1, "poison": 2, "delay": 3}
OK, ERR_INVALID, ERR_NOT_INIT, ERR_TOO_LARGE, ERR_UNSUPPORTED, ERR_OCCUPANCY, ERR_CUDA, ERR_TIMEOUT = range(8)

_lib = None


class LLBufferStatus(ctypes.Structure):
    """llar_llbuffer_status (include/llar_llbuffer.h)."""
    _fields_ = [("code", ctypes.c_uint), ("rank", ctypes.c_int), ("epoch", ctypes.c_ulonglong)]


class LLBufferDesc(ctypes.Structure):
    """llar_llbuffer (include/llar_llbuffer.h), field for field."""
    _fields_ = [("nranks", ctypes.c_int), ("reserved", ctypes.c_int), ("bytes", ctypes.c_size_t),
                ("timeout_ns", ctypes.c_ulonglong),
                ("ll", ctypes.c_void_p), ("ll_rank_stride", ctypes.c_size_t),
                ("ll_slot_stride", ctypes.c_size_t), ("ll_words", ctypes.c_size_t),
                ("sen", ctypes.c_void_p), ("sen_rank_stride", ctypes.c_size_t),
                ("sen_slot_stride", ctypes.c_size_t), ("sen_src_stride", ctypes.c_size_t),
                ("sen_vecs", ctypes.c_size_t),
                ("ll128", ctypes.c_void_p), ("ll128_rank_stride", ctypes.c_size_t),
                ("ll128_slot_stride", ctypes.c_size_t), ("ll128_lines", ctypes.c_size_t),
                ("epoch", ctypes.c_void_p), ("done_count", ctypes.c_void_p),
                ("abort_word", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("status_host", ctypes.c_void_p)]


class LlarError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (status {code})")


def lib():
    """The loaded libllar.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m tp_allreduce_persistent_b300.build` (no CPU fallback exists)")
    L = ctypes.CDLL(LIB_PATH)
    c_int, c_size, c_vp, c_ull = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_ulonglong
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "llar_init": (c_int, [c_int, c_int, c_size]),
        "llar_destroy": (c_int, []),
        "llar_allreduce": (c_int, [pp, pp, c_size, c_int, c_vp]),
        "llar_allreduce_iters": (c_int, [pp, pp, c_size, c_int, c_int, c_size, c_size, ctypes.c_float, c_vp]),
        "llar_allreduce_host": (c_int, [c_vp, c_vp, c_size, c_int, c_vp]),
        "llar_reduce_scatter": (c_int, [pp, pp, c_size, c_int, c_vp]),
        "llar_all_gather": (c_int, [pp, pp, c_size, c_int, c_vp]),
        "llar_sendrecv": (c_int, [pp, pp, ctypes.POINTER(c_int), c_size, c_int, c_int, c_size, c_size, c_vp]),
        "llar_allreduce_noalloc": (c_int, [pp, pp, c_size, c_int, c_int, c_vp]),
        "llar_get_status": (c_int, [ctypes.POINTER(c_int), ctypes.POINTER(c_int), ctypes.POINTER(c_ull)]),
        "llar_reset": (c_int, [c_vp]),
        "llar_set_timeout_ns": (None, [c_ull]),
        "llar_set_launch": (c_int, [c_int, c_int]),
        "llar_set_sentinel_chunk": (c_int, [c_size]),
        "llar_debug_inject": (c_int, [c_int, c_int]),
        "llar_sol_probe": (c_int, [ctypes.POINTER(ctypes.c_double)] * 3),
        "llar_sol_probe_detail": (c_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int),
                                          ctypes.POINTER(c_int), ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(c_int), ctypes.POINTER(c_int),
                                          ctypes.POINTER(c_int)]),
        "llar_staging": (c_int, [c_int, ctypes.POINTER(c_vp), ctypes.POINTER(c_size), ctypes.POINTER(c_size)]),
        "llar_layout": (c_int, [c_int, c_int, c_int, c_size, ctypes.POINTER(c_size),
                                ctypes.POINTER(c_size), ctypes.POINTER(c_size)]),
        "llar_select_protocol": (c_int, [c_int, c_int, c_size]),
        "llar_select_protocol_host": (c_int, [c_int, c_int, c_size]),
        "llar_select_protocol_segment": (c_int, [c_int, c_int, c_int, c_size]),
        "llar_select_protocol_iters": (c_int, [c_int, c_int, c_size, c_int, c_int, c_int]),
        "llar_set_auto_nondeterministic": (c_int, [c_int]),
        "llar_epoch": (c_ull, []),
        "llar_sol_bound_us": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
        "llar_sol_probe_placed": (c_int, [ctypes.POINTER(ctypes.c_double)] * 3 + [ctypes.POINTER(c_int)]),
        "llar_ll_placement": (c_int, [ctypes.POINTER(c_int)]),
        "llar_last_launch": (c_int, [ctypes.POINTER(c_int)] * 4),
        "llar_host_register": (c_int, [c_vp, c_size]),
        "llar_host_unregister": (c_int, [c_vp]),
        "llar_debug_launch_shape": (c_int, [c_int, c_int, c_size, c_int, c_int, c_int, c_size,
                                            ctypes.POINTER(c_int), ctypes.POINTER(c_int)]),
        "llar_strerror": (ctypes.c_char_p, [c_int]),
        "llar_debug_poll_stats": (c_int, [ctypes.POINTER(c_ull), c_int]),
        "llar_llbuffer_create": (c_int, [c_int, c_size, ctypes.POINTER(LLBufferDesc)]),
        "llar_llbuffer_destroy": (c_int, [ctypes.POINTER(LLBufferDesc)]),
        "llar_llbuffer_get_status": (c_int, [ctypes.POINTER(LLBufferDesc), ctypes.POINTER(c_int),
                                             ctypes.POINTER(c_ull)]),
        "llar_llbuffer_reset": (c_int, [ctypes.POINTER(LLBufferDesc), c_vp]),
        "llar_llbuffer_set_timeout_ns": (c_int, [ctypes.POINTER(LLBufferDesc), c_ull]),
        "llar_llbuffer_epoch": (c_int, [ctypes.POINTER(LLBufferDesc), ctypes.POINTER(c_ull)]),
        "llar_llbuffer_probe_wait": (c_int, [ctypes.POINTER(LLBufferDesc), c_int, c_int, c_ull, c_size, c_vp]),
        "llar_llbuffer_allreduce": (c_int, [ctypes.POINTER(LLBufferDesc), pp, pp, c_size, c_int, c_int,
                                            c_int, c_vp]),
        "llar_fused_linear_allreduce": (c_int, [ctypes.POINTER(LLBufferDesc), pp, pp, pp, c_int, c_int,
                                                c_int, c_int, c_vp]),
        "llar_linear_partials": (c_int, [pp, pp, pp, c_int, c_int, c_int, c_int, c_int, c_vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(code, what):
    if code != OK:
        raise LlarError(code, what)
    return code


def _enum(table, value):
    return table[value] if isinstance(value, str) else int(value)


def _ptr(x):
    return x.data_ptr() if hasattr(x, "data_ptr") else int(x)


_PTR_ARRAY_TYPES = {}


def _ptr_array(xs):
    """Host array of the N pointers (tensors or integers). Marshalling only:
    a call from Python pays this per pointer array, so the array type is
    kept per length and tensors take the direct path."""
    n = len(xs)
    t = _PTR_ARRAY_TYPES.get(n)
    if t is None:
        t = _PTR_ARRAY_TYPES[n] = ctypes.c_void_p * n
    try:
        return t(*[x.data_ptr() for x in xs])
    except AttributeError:
        return t(*[_ptr(x) for x in xs])


_raw_stream = None


def _stream(stream):
    """cudaStream_t of `stream`; None means torch's current stream."""
    global _raw_stream
    if stream is None:
        if _raw_stream is None:
            import torch
            if not torch.cuda.is_available():
                return 0
            getter = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
            torch.cuda.init()
            _raw_stream = (lambda: getter(device())) if getter else \
                (lambda: torch.cuda.current_stream().cuda_stream)
        return _raw_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def strerror(code):
    return lib().llar_strerror(int(code)).decode()


def llar_init(nranks, dtype, max_bytes):
    _check(lib().llar_init(int(nranks), _enum(DTYPES, dtype), int(max_bytes)), "llar_init")


def llar_destroy():
    _check(lib().llar_destroy(), "llar_destroy")


def llar_allreduce(ins, outs, count=None, protocol="auto", stream=None):
    """One AllReduce: outs[r] = sum over q of ins[q] (lists of N device tensors)."""
    if count is None:
        count = ins[0].numel()
    _check(lib().llar_allreduce(_ptr_array(ins), _ptr_array(outs), int(count),
                                _enum(PROTOCOLS, protocol), ctypes.c_void_p(_stream(stream))),
           "llar_allreduce")


def llar_allreduce_iters(ins, outs, count, protocol, iters, in_stride=0, out_stride=0,
                         chain_scale=0.0, stream=None):
    """`iters` AllReduces in one persistent launch (strides in elements)."""
    _check(lib().llar_allreduce_iters(_ptr_array(ins), _ptr_array(outs), int(count),
                                      _enum(PROTOCOLS, protocol), int(iters), int(in_stride),
                                      int(out_stride), float(chain_scale),
                                      ctypes.c_void_p(_stream(stream))),
           "llar_allreduce_iters")


def llar_reduce_scatter(ins, outs, count, protocol="auto", stream=None):
    """outs[r] = rank-order sum of segment r of every ins[q] (count = full length)."""
    _check(lib().llar_reduce_scatter(_ptr_array(ins), _ptr_array(outs), int(count),
                                     _enum(PROTOCOLS, protocol), ctypes.c_void_p(_stream(stream))),
           "llar_reduce_scatter")


def llar_all_gather(ins, outs, count, protocol="auto", stream=None):
    """outs[r] = concatenation of every rank's segment ins[q] (count = full length)."""
    _check(lib().llar_all_gather(_ptr_array(ins), _ptr_array(outs), int(count),
                                 _enum(PROTOCOLS, protocol), ctypes.c_void_p(_stream(stream))),
           "llar_all_gather")


def llar_sendrecv(sends, recvs, dst, count, protocol="auto", iters=1, send_stride=0, recv_stride=0,
                  stream=None):
    """recvs[dst[r]] = sends[r] for every r with dst[r] >= 0 (None: no buffer)."""
    n = len(dst)
    d = (ctypes.c_int * n)(*[int(v) for v in dst])
    _check(lib().llar_sendrecv(_ptr_array([0 if t is None else t for t in sends]),
                               _ptr_array([0 if t is None else t for t in recvs]), d, int(count),
                               _enum(PROTOCOLS, protocol), int(iters), int(send_stride), int(recv_stride),
                               ctypes.c_void_p(_stream(stream))),
           "llar_sendrecv")


def llar_allreduce_host(in_host, out_host, count, protocol="auto", stream=None):
    """AllReduce of host [N][count] arrays (tensors or raw host pointers)."""
    _check(lib().llar_allreduce_host(ctypes.c_void_p(_ptr(in_host)), ctypes.c_void_p(_ptr(out_host)),
                                     int(count), _enum(PROTOCOLS, protocol),
                                     ctypes.c_void_p(_stream(stream))),
           "llar_allreduce_host")


def llar_host_register(buf, nbytes=None):
    """Register a pinned host buffer (tensor or raw pointer + nbytes) for llar_allreduce_host."""
    if nbytes is None:
        nbytes = buf.numel() * buf.element_size()
    _check(lib().llar_host_register(ctypes.c_void_p(_ptr(buf)), int(nbytes)), "llar_host_register")


def llar_host_unregister(buf):
    _check(lib().llar_host_unregister(ctypes.c_void_p(_ptr(buf))), "llar_host_unregister")


def llar_allreduce_noalloc(ins, outs, count, nranks, dtype, stream=None):
    """LL AllReduce with library-internal static staging (no allocation, no init)."""
    _check(lib().llar_allreduce_noalloc(_ptr_array(ins), _ptr_array(outs), int(count), int(nranks),
                                        _enum(DTYPES, dtype), ctypes.c_void_p(_stream(stream))),
           "llar_allreduce_noalloc")


def llar_debug_poll_stats(reset=True):
    """(thread polling rounds, line loads, waits, lines awaited) counted by
    the poll-counting build since the last reset; raises LlarError
    (ERR_UNSUPPORTED) in the regular build."""
    out = (ctypes.c_ulonglong * 4)()
    _check(lib().llar_debug_poll_stats(out, 1 if reset else 0), "llar_debug_poll_stats")
    return tuple(int(v) for v in out)


def llar_get_status():
    """(code, rank, cta, epoch) of the device status word."""
    r, c, e = ctypes.c_int(), ctypes.c_int(), ctypes.c_ulonglong()
    code = lib().llar_get_status(ctypes.byref(r), ctypes.byref(c), ctypes.byref(e))
    return code, r.value, c.value, e.value


def llar_reset(stream=None):
    _check(lib().llar_reset(ctypes.c_void_p(_stream(stream))), "llar_reset")


def llar_set_timeout_ns(ns):
    lib().llar_set_timeout_ns(int(ns))


def llar_set_launch(ctas_per_rank=0, threads=0):
    _check(lib().llar_set_launch(int(ctas_per_rank), int(threads)), "llar_set_launch")


def llar_set_sentinel_chunk(nbytes):
    _check(lib().llar_set_sentinel_chunk(int(nbytes)), "llar_set_sentinel_chunk")


def llar_debug_inject(rank, mode):
    _check(lib().llar_debug_inject(int(rank), _enum(INJECT, mode)), "llar_debug_inject")


def llar_sol_probe():
    """(l2_round_trip_us, write_us, speed_of_light_us)."""
    a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(lib().llar_sol_probe(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "llar_sol_probe")
    return a.value, b.value, c.value


def llar_ll_placement():
    """1 if this context runs long LL launches in clusters of N blocks (chosen
    by timing both at llar_init), else 0."""
    v = ctypes.c_int()
    _check(lib().llar_ll_placement(ctypes.byref(v)), "llar_ll_placement")
    return v.value


def llar_sol_probe_placed():
    """(l2_rt_us, write_us, sol_us, pairs) at the worst pair of the rank CTAs
    placed by a launch shaped like the most recent AllReduce."""
    a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    n = ctypes.c_int()
    _check(lib().llar_sol_probe_placed(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), ctypes.byref(n)),
           "llar_sol_probe_placed")
    return a.value, b.value, c.value, n.value


def llar_sol_bound_us(l2_rt_us, write_us):
    """Speed-of-light bound 2 * L2 round trip + one write (host arithmetic)."""
    return float(lib().llar_sol_bound_us(float(l2_rt_us), float(write_us)))


def llar_sol_probe_detail():
    """Per-SM chase latencies and per-pair ping-pong round trips (ns)."""
    chase = (ctypes.c_double * 256)()
    csm = (ctypes.c_int * 256)()
    rt = (ctypes.c_double * 128)()
    sa = (ctypes.c_int * 128)()
    sb = (ctypes.c_int * 128)()
    nc, npair = ctypes.c_int(), ctypes.c_int()
    _check(lib().llar_sol_probe_detail(chase, csm, ctypes.byref(nc), rt, sa, sb, ctypes.byref(npair)),
           "llar_sol_probe_detail")
    return {"chase_ns": list(chase[:nc.value]), "chase_smid": list(csm[:nc.value]),
            "rt_ns": list(rt[:npair.value]), "smid_a": list(sa[:npair.value]),
            "smid_b": list(sb[:npair.value])}


def llar_staging(protocol):
    """(device pointer, rank stride bytes, bytes used per rank) of a protocol's staging."""
    p, s, u = ctypes.c_void_p(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().llar_staging(_enum(PROTOCOLS, protocol), ctypes.byref(p), ctypes.byref(s),
                              ctypes.byref(u)), "llar_staging")
    return p.value, s.value, u.value


def llar_layout(protocol, dtype, nranks, count):
    """(line bytes, data elements per line, staging bytes per rank) — host only."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().llar_layout(_enum(PROTOCOLS, protocol), _enum(DTYPES, dtype), int(nranks), int(count),
                             ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "llar_layout")
    return a.value, b.value, c.value


def llar_select_protocol(nranks, dtype, count):
    return PROTOCOL_NAMES[lib().llar_select_protocol(int(nranks), _enum(DTYPES, dtype), int(count))]


def llar_select_protocol_iters(nranks, dtype, count, iters, chained=False, nondeterministic=False):
    """AUTO's choice for llar_allreduce_iters (default LL capacity)."""
    return PROTOCOL_NAMES[lib().llar_select_protocol_iters(int(nranks), _enum(DTYPES, dtype), int(count),
                                                           int(iters), int(bool(chained)),
                                                           int(bool(nondeterministic)))]


def llar_set_auto_nondeterministic(allow):
    """Let AUTO pick the LL128 direct protocol where it measured fastest."""
    _check(lib().llar_set_auto_nondeterministic(int(bool(allow))), "llar_set_auto_nondeterministic")


def llar_select_protocol_segment(reduce_scatter, nranks, dtype, count):
    """AUTO's choice for llar_reduce_scatter (True) or llar_all_gather (False)."""
    return PROTOCOL_NAMES[lib().llar_select_protocol_segment(int(bool(reduce_scatter)), int(nranks),
                                                             _enum(DTYPES, dtype), int(count))]


def llar_select_protocol_host(nranks, dtype, count):
    """AUTO's choice for llar_allreduce_host on pinned, device-addressable buffers."""
    return PROTOCOL_NAMES[lib().llar_select_protocol_host(int(nranks), _enum(DTYPES, dtype), int(count))]


def llar_epoch():
    return int(lib().llar_epoch())


def llar_last_launch():
    """(protocol name, CTAs per rank, threads per CTA, iterations) of the latest launch."""
    v = [ctypes.c_int() for _ in range(4)]
    lib().llar_last_launch(*[ctypes.byref(x) for x in v])
    return PROTOCOL_NAMES.get(v[0].value, v[0].value), v[1].value, v[2].value, v[3].value


def llar_debug_launch_shape(nranks, dtype, count, protocol, chained=False, sms=148, chunk_bytes=64 << 10):
    """(CTAs per rank, threads per CTA) the launch-shape rule picks; host arithmetic only.
    chained: 0/False a loop of AllReduces, 1/True a chain, 2 one AllReduce per launch."""
    g, t = ctypes.c_int(), ctypes.c_int()
    _check(lib().llar_debug_launch_shape(int(nranks), _enum(DTYPES, dtype), int(count), _enum(PROTOCOLS, protocol),
                                         int(chained), int(sms), int(chunk_bytes), ctypes.byref(g),
                                         ctypes.byref(t)), "llar_debug_launch_shape")
    return g.value, t.value


# ------------------------------------------------------------ LL buffer API
class LLBuffer:
    """An llar_llbuffer descriptor (include/llar_llbuffer.h) and its calls.

    Owns the device staging until close(); usable as a context manager."""

    def __init__(self, nranks, nbytes):
        self.desc = LLBufferDesc()
        _check(lib().llar_llbuffer_create(int(nranks), int(nbytes), ctypes.byref(self.desc)),
               "llar_llbuffer_create")

    def close(self):
        if self.desc.ll:
            _check(lib().llar_llbuffer_destroy(ctypes.byref(self.desc)), "llar_llbuffer_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def nranks(self):
        return self.desc.nranks

    def status(self):
        """(code, rank, epoch) of the descriptor's error record."""
        r, e = ctypes.c_int(), ctypes.c_ulonglong()
        code = lib().llar_llbuffer_get_status(ctypes.byref(self.desc), ctypes.byref(r), ctypes.byref(e))
        return code, r.value, e.value

    def reset(self, stream=None):
        _check(lib().llar_llbuffer_reset(ctypes.byref(self.desc), ctypes.c_void_p(_stream(stream))),
               "llar_llbuffer_reset")

    def set_timeout_ns(self, ns):
        _check(lib().llar_llbuffer_set_timeout_ns(ctypes.byref(self.desc), int(ns)),
               "llar_llbuffer_set_timeout_ns")

    def epoch(self):
        """Exchanges completed so far (the device counter; synchronises the device)."""
        e = ctypes.c_ulonglong()
        _check(lib().llar_llbuffer_epoch(ctypes.byref(self.desc), ctypes.byref(e)), "llar_llbuffer_epoch")
        return e.value

    def probe_wait(self, rank, src, epoch, word, stream=None):
        _check(lib().llar_llbuffer_probe_wait(ctypes.byref(self.desc), int(rank), int(src), int(epoch),
                                              int(word), ctypes.c_void_p(_stream(stream))),
               "llar_llbuffer_probe_wait")

    def allreduce(self, ins, outs, count, dtype, protocol="ll", iters=1, stream=None):
        _check(lib().llar_llbuffer_allreduce(ctypes.byref(self.desc), _ptr_array(ins), _ptr_array(outs),
                                             int(count), _enum(DTYPES, dtype), _enum(PROTOCOLS, protocol),
                                             int(iters), ctypes.c_void_p(_stream(stream))),
               "llar_llbuffer_allreduce")

    def fused_linear_allreduce(self, xs, ws, outs, m, k, h, dtype, stream=None):
        _check(lib().llar_fused_linear_allreduce(ctypes.byref(self.desc), _ptr_array(xs), _ptr_array(ws),
                                                 _ptr_array(outs), int(m), int(k), int(h),
                                                 _enum(DTYPES, dtype), ctypes.c_void_p(_stream(stream))),
               "llar_fused_linear_allreduce")


def llar_linear_partials(xs, ws, ps, m, k, h, dtype, stream=None):
    """ps[r] = rounded x[r] @ w[r] (the unfused layer's GEMV launch)."""
    _check(lib().llar_linear_partials(_ptr_array(xs), _ptr_array(ws), _ptr_array(ps), len(xs), int(m),
                                      int(k), int(h), _enum(DTYPES, dtype), ctypes.c_void_p(_stream(stream))),
           "llar_linear_partials")


# C-named entry points of the LL buffer API (the LLBuffer methods wrap them)
def llar_llbuffer_create(nranks, nbytes):
    return LLBuffer(nranks, nbytes)


def llar_llbuffer_destroy(buf):
    buf.close()


def llar_llbuffer_get_status(buf):
    return buf.status()


def llar_llbuffer_reset(buf, stream=None):
    buf.reset(stream)


def llar_llbuffer_set_timeout_ns(buf, ns):
    buf.set_timeout_ns(ns)


def llar_llbuffer_epoch(buf):
    return buf.epoch()


def llar_llbuffer_allreduce(buf, ins, outs, count, dtype, protocol="ll", iters=1, stream=None):
    buf.allreduce(ins, outs, count, dtype, protocol, iters, stream)


def llar_fused_linear_allreduce(buf, xs, ws, outs, m, k, h, dtype, stream=None):
    buf.fused_linear_allreduce(xs, ws, outs, m, k, h, dtype, stream)


def llar_llbuffer_probe_wait(buf, rank, src, epoch, word, stream=None):
    buf.probe_wait(rank, src, epoch, word, stream)
