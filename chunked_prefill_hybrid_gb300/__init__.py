"""GB300 (sm_103a) hybrid-batch forward: one prefill chunk plus piggybacked
decodes through a LLaMA-style decoder-layer stack, behind a C ABI
(include/hb.h, libhb.so) with a thin ctypes binding (native.py) and a host
decode-maximal scheduler (sched.py, libhb's hb_sched_* calls)."""
