"""CPU oracles for WISE paged decode attention (test infrastructure only).

wise_oracle.py is the numpy float64 definition; wise_oracle.cpp (loaded
through cpp_oracle.py) is the same definition as plain C++ in fp32, with a
double instantiation of the same code that bounds its rounding.  Only the
tests, the smoke check and the benchmark's CPU-baseline leg use them."""
