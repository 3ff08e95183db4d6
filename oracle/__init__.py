"""CPU fp64 oracle for the TurboQuant packed-KV writer and paged decode.

Test infrastructure only: the product path never imports this package.
"""
