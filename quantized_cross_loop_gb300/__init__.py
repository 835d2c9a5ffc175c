"""GB300-native FlashLoop packed-KV path: INT4 base + cross-loop residual codec,
residual-chain reconstruction and packed-KV GQA decode attention, all in
hand-written sm_103a CUDA behind the C ABI declared in include/kvq.h.

The binding (``kvq``) loads the in-tree ``libkvq.so`` on first use and raises if
it is missing: there is no CPU fallback.
"""
